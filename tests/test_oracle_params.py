"""Pins of the oracle's parameter counts against the page's closed forms and its printed figures.

Page: "Как устроен Olmo-core 3: обучение больших MoE-моделей", sections
"Как задаётся конфигурация MoE" (formulas) and "Как сравнивали и что
получилось" (the 8 -> 128 expert-pool figures).
"""
import os

import pytest

from oracle import moe_ref as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_kv(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            out[k] = float(v)
    return out


def _read_table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


@pytest.mark.parametrize("row", _read_table("param_counts.txt"), ids=lambda r: r[0])
def test_param_counts_closed_form(row):
    name, D, L, E, k, h, router, total, active, proj = row[0], *map(int, row[1:])
    cfg = ref.OracleConfig(d_model=D, num_experts=E, top_k=k, hidden_size=h, latent_dim=L)
    assert ref.router_params(cfg) == router
    assert ref.num_params(cfg) == total
    assert ref.num_active_params(cfg) == active
    assert ref.latent_proj_params(cfg) == proj


def test_router_bias_and_up_factor():
    cfg = ref.OracleConfig(d_model=64, num_experts=10, top_k=2, hidden_size=32, router_bias=True)
    assert ref.router_params(cfg) == 64 * 10 + 10
    # (up_factor + 1) * d * h: 3 for the gated activations, 2 for a plain one
    assert ref.expert_params_each(cfg, "swiglu") == 3 * 64 * 32
    assert ref.expert_params_each(cfg, "gpt_oss_swiglu") == 3 * 64 * 32
    assert ref.expert_params_each(cfg, "gelu") == 2 * 64 * 32
    # shared modules add to total and active alike
    assert ref.num_params(cfg, shared_params=7) == ref.num_params(cfg) + 7
    assert ref.num_active_params(cfg, shared_params=7) == ref.num_active_params(cfg) + 7


def test_expert_pool_scaling_figures():
    """The page's 8 -> 128 expert figures are consistent with total = base + E*P, active = base + k*P.

    From the two totals: P = (47B - 4.6B) / 120, base = 4.6B - 8P, so active = base + 4P ~ 3.19B,
    which the page prints as ~3.2B.  The oracle's formulas must have the same
    affine structure in the expert count.
    """
    g = _read_kv("expert_pool_scaling.txt")
    e0, e1, k = int(g["experts_before"]), int(g["experts_after"]), int(g["top_k"])
    per_expert = (g["total_after"] - g["total_before"]) / (e1 - e0)
    base = g["total_before"] - e0 * per_expert
    predicted_active = base + k * per_expert
    assert abs(predicted_active - g["active_approx"]) / g["active_approx"] < g["rel_tolerance"]

    # Same structure in the oracle, for an arbitrary layer shape.
    def cfg(E):
        return ref.OracleConfig(d_model=1536, num_experts=E, top_k=k, hidden_size=768)

    P = (ref.num_params(cfg(e1)) - ref.num_params(cfg(e0))) // (e1 - e0)
    # each added expert brings its MLP and one router row of d_model weights
    assert P == ref.expert_params_each(cfg(e0)) + 1536
    Pe = ref.expert_params_each(cfg(e0))
    # active = total minus the (E - k) experts that a token does not use
    assert ref.num_active_params(cfg(e0)) == ref.num_params(cfg(e0)) - (e0 - k) * Pe
    assert ref.num_active_params(cfg(e1)) == ref.num_params(cfg(e1)) - (e1 - k) * Pe
    # only the router's rows make the active count grow with the pool
    assert ref.num_active_params(cfg(e1)) - ref.num_active_params(cfg(e0)) == (e1 - e0) * 1536


def test_latent_counts_use_latent_dim():
    """Experts are built with d_model = latent_dim, so the latent layer's expert count uses L."""
    dense = ref.OracleConfig(d_model=2048, num_experts=4, top_k=1, hidden_size=256)
    lat = ref.OracleConfig(d_model=4096, num_experts=4, top_k=1, hidden_size=256, latent_dim=2048)
    assert ref.num_params(lat) - ref.router_params(lat) == ref.num_params(dense) - ref.router_params(dense)
