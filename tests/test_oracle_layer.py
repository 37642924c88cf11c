"""Pins of the oracle's whole layer: dense reductions, latent identity, library RMSNorm / SiLU.

Page: "Как устроен Olmo-core 3: обучение больших MoE-моделей", sections
"Латентная проекция экспертов" (prepare_routed_input / restore_routed_output,
bias-free RMSNorm), "Маршрутизация: как роутер выбирает экспертов" and
"Вычисления экспертов и точность" / "SwiGLU с квантизацией" (the SwiGLU
expert and the split into up and gate).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import moe_ref as ref


def _weights(D, L, E, h, seed, latent=False, router_scale=1.0):
    g = np.random.default_rng(seed)
    ups = g.standard_normal((E, h, L)) * 0.2
    gates = g.standard_normal((E, h, L)) * 0.2
    outs = g.standard_normal((E, L, h)) * 0.2
    w = ref.OracleWeights(w_router=g.standard_normal((E, D)) * router_scale,
                          expert=lambda e: (ups[e], gates[e], outs[e]))
    if latent:
        w.w_down_latent = g.standard_normal((L, D)) * 0.2
        w.w_up_latent = g.standard_normal((D, L)) * 0.2
    return w, ups, gates, outs


def _torch_swiglu(x, up, gate, out):
    xt = torch.from_numpy(x)
    return F.linear(F.silu(F.linear(xt, torch.from_numpy(gate))) * F.linear(xt, torch.from_numpy(up)),
                    torch.from_numpy(out)).numpy()


def test_softmax_all_experts_is_dense_mixture():
    T, D, E, h = 12, 16, 5, 8
    w, ups, gates, outs = _weights(D, D, E, h, seed=1)
    x = np.random.default_rng(2).standard_normal((T, D))
    cfg = ref.OracleConfig(d_model=D, num_experts=E, top_k=E, hidden_size=h, gating=ref.GATING_SOFTMAX)
    res = ref.layer_forward(cfg, x, w)
    s = torch.softmax(torch.from_numpy(x @ w.w_router.T), dim=1).numpy()
    dense = sum(s[:, e:e + 1] * _torch_swiglu(x, ups[e], gates[e], outs[e]) for e in range(E))
    np.testing.assert_allclose(res.out, dense, rtol=1e-11, atol=1e-13)


def test_single_expert_is_dense_swiglu_mlp():
    T, D, h = 9, 24, 12
    w, ups, gates, outs = _weights(D, D, 1, h, seed=3)
    x = np.random.default_rng(4).standard_normal((T, D))
    cfg = ref.OracleConfig(d_model=D, num_experts=1, top_k=1, hidden_size=h, gating=ref.GATING_SOFTMAX)
    res = ref.layer_forward(cfg, x, w)
    np.testing.assert_allclose(res.out, _torch_swiglu(x, ups[0], gates[0], outs[0]), rtol=1e-12, atol=1e-14)


def test_topk_layer_matches_per_token_sum():
    """Any k: out[t] = sum_j w[t,j] * MLP_{idx[t,j]}(x[t]) (no permutation involved)."""
    T, D, E, h, k = 20, 16, 6, 8, 3
    w, ups, gates, outs = _weights(D, D, E, h, seed=5)
    x = np.random.default_rng(6).standard_normal((T, D))
    cfg = ref.OracleConfig(d_model=D, num_experts=E, top_k=k, hidden_size=h, gating=ref.GATING_SIGMOID,
                           normalize_expert_weights=1.0)
    res = ref.layer_forward(cfg, x, w)
    want = np.zeros((T, D))
    for t in range(T):
        for j in range(k):
            e = res.routing.idx[t, j]
            want[t] += res.routing.weights[t, j] * _torch_swiglu(x[t:t + 1], ups[e], gates[e], outs[e])[0]
    np.testing.assert_allclose(res.out, want, rtol=1e-11, atol=1e-13)


def test_identity_latent_equals_plain_layer():
    T, D, E, h, k = 10, 16, 4, 8, 2
    w, *_ = _weights(D, D, E, h, seed=7)
    x = np.random.default_rng(8).standard_normal((T, D))
    plain = ref.OracleConfig(d_model=D, num_experts=E, top_k=k, hidden_size=h, gating=ref.GATING_SIGMOID)
    lat = ref.OracleConfig(d_model=D, num_experts=E, top_k=k, hidden_size=h, gating=ref.GATING_SIGMOID,
                           latent_dim=D, up_proj_norm=False)
    wl = ref.OracleWeights(w_router=w.w_router, expert=w.expert, w_down_latent=np.eye(D), w_up_latent=np.eye(D))
    np.testing.assert_allclose(ref.layer_forward(lat, x, wl).out, ref.layer_forward(plain, x, w).out,
                               rtol=1e-13, atol=1e-15)


def test_rms_norm_matches_library():
    z = np.random.default_rng(9).standard_normal((7, 32)) * 3
    got = ref.rms_norm(z, 1e-6)
    want = F.rms_norm(torch.from_numpy(z), (32,), eps=1e-6).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-13)
    gamma = np.random.default_rng(10).standard_normal(32)
    want_g = F.rms_norm(torch.from_numpy(z), (32,), weight=torch.from_numpy(gamma), eps=1e-6).numpy()
    np.testing.assert_allclose(ref.rms_norm(z, 1e-6, gamma), want_g, rtol=1e-13)


def test_silu_matches_library():
    g = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(ref.silu(g), F.silu(torch.from_numpy(g)).numpy(), rtol=1e-13, atol=1e-300)


def test_latent_layer_restores_through_norm_and_up_projection():
    T, D, L, E, h, k = 8, 24, 16, 4, 8, 2
    w, *_ = _weights(D, L, E, h, seed=11, latent=True)
    x = np.random.default_rng(12).standard_normal((T, D))
    cfg = ref.OracleConfig(d_model=D, num_experts=E, top_k=k, hidden_size=h, latent_dim=L,
                           gating=ref.GATING_SIGMOID)
    res = ref.layer_forward(cfg, x, w)
    assert res.x_routed.shape == (T, L) and res.out.shape == (T, D)
    np.testing.assert_allclose(res.x_routed, (torch.from_numpy(x) @ torch.from_numpy(w.w_down_latent).T).numpy(),
                               rtol=1e-12)
    n = F.rms_norm(torch.from_numpy(res.z), (L,), eps=cfg.rms_eps)
    np.testing.assert_allclose(res.out, (n @ torch.from_numpy(w.w_up_latent).T).numpy(), rtol=1e-11, atol=1e-13)
    # the router reads x, not the latent projection: changing W_down leaves the routing alone
    w2 = ref.OracleWeights(w_router=w.w_router, expert=w.expert, w_down_latent=w.w_down_latent * -3.0,
                           w_up_latent=w.w_up_latent)
    np.testing.assert_array_equal(ref.layer_forward(cfg, x, w2).routing.idx, res.routing.idx)


def test_layer_on_token_subset_equals_rows_of_full_layer():
    """Tokens are independent: the layer on a subset equals those rows of the full layer."""
    T, D, E, h, k = 30, 16, 6, 8, 2
    w, *_ = _weights(D, D, E, h, seed=13)
    x = np.random.default_rng(14).standard_normal((T, D))
    cfg = ref.OracleConfig(d_model=D, num_experts=E, top_k=k, hidden_size=h, gating=ref.GATING_TOPK_SOFTMAX)
    full = ref.layer_forward(cfg, x, w).out
    sub = [3, 17, 29, 0]
    np.testing.assert_allclose(ref.layer_forward(cfg, x[sub], w).out, full[sub], rtol=1e-12, atol=1e-14)
