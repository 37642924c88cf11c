"""Pins of the oracle's backward: the hand-derived gradients of the SwiGLU expert, the grouped
experts and the combine against central finite differences of the forward oracle (float64,
tiny sizes), and silu' against torch autograd."""
import numpy as np
import torch

from oracle import moe_ref as ref


def _fd(f, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + eps
        fp = f()
        x[i] = old - eps
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * eps)
    return g


def test_silu_grad_matches_autograd():
    g = torch.linspace(-20, 20, 401, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.silu(g).sum().backward()
    np.testing.assert_allclose(ref.silu_grad(g.detach().numpy()), g.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_swiglu_mlp_backward_finite_differences():
    rng = np.random.default_rng(0)
    n, L, h = 3, 5, 4
    rows, wu, wg = rng.standard_normal((n, L)), rng.standard_normal((h, L)), rng.standard_normal((h, L))
    wo, probe = rng.standard_normal((L, h)), rng.standard_normal((n, L))
    loss = lambda: float((ref.swiglu_mlp(rows, wu, wg, wo) * probe).sum())   # noqa: E731
    d_rows, dwu, dwg, dwo, h_act = ref.swiglu_mlp_backward(rows, wu, wg, wo, probe)
    for got, arr in ((d_rows, rows), (dwu, wu), (dwg, wg), (dwo, wo)):
        np.testing.assert_allclose(got, _fd(loss, arr), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(h_act, ref.silu(rows @ wg.T) * (rows @ wu.T), rtol=1e-14)


def test_experts_and_combine_backward_finite_differences():
    rng = np.random.default_rng(1)
    T, L, E, h, k = 6, 4, 3, 3, 2
    ups, gates, outs = rng.standard_normal((E, h, L)), rng.standard_normal((E, h, L)), rng.standard_normal((E, L, h))
    x = rng.standard_normal((T, L))
    idx = np.array([[0, 2], [1, 0], [2, 1], [0, 1], [2, 0], [1, 2]])
    w = rng.random((T, k))
    perm = ref.permute(idx, E)
    cfg = ref.OracleConfig(d_model=L, num_experts=E, top_k=k, hidden_size=h)
    expert = lambda e: (ups[e], gates[e], outs[e])   # noqa: E731
    probe = rng.standard_normal((T, L))

    def loss():
        y = ref.expert_outputs(cfg, x, perm, expert)
        return float((ref.combine(y, perm.scatter_pos, w) * probe).sum())

    y = ref.expert_outputs(cfg, x, perm, expert)
    dy, dw = ref.combine_backward(probe, y, perm.scatter_pos, w)
    np.testing.assert_allclose(dw, _fd(loss, w), rtol=1e-6, atol=1e-8)
    dx, grads = ref.experts_backward(cfg, x, perm, expert, dy)
    np.testing.assert_allclose(dx, _fd(loss, x), rtol=1e-6, atol=1e-8)
    for e in range(E):
        np.testing.assert_allclose(grads[e][0], _fd(loss, ups[e]), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(grads[e][1], _fd(loss, gates[e]), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(grads[e][2], _fd(loss, outs[e]), rtol=1e-6, atol=1e-8)


import pytest  # noqa: E402


@pytest.mark.parametrize("gating,extra", [
    (ref.GATING_SOFTMAX, dict(normalize_expert_weights=1.0)),
    (ref.GATING_TOPK_SOFTMAX, dict(restore_weight_scale=True)),
    (ref.GATING_SIGMOID, dict(sigmoid_stability_epsilon=1e-3, normalize_expert_weights=1.0, expert_weight_scale=2.0)),
    (ref.GATING_SIGMOID, dict(normalize_expert_weights=2.0, original_top_k=8)),
    (ref.GATING_SOFTMAX, dict()),
])
def test_router_backward_finite_differences(gating, extra):
    rng = np.random.default_rng(3)
    T, D, E, k = 4, 5, 6, 2
    x, w, b = rng.standard_normal((T, D)), rng.standard_normal((E, D)) * 0.5, rng.standard_normal(E) * 0.1
    sb = rng.standard_normal(E)
    cfg = ref.OracleConfig(d_model=D, num_experts=E, top_k=k, hidden_size=4, gating=gating, router_bias=True,
                           has_score_bias=True, **extra)
    idx = ref.route(cfg, x, w, b, sb).idx               # the choice is held fixed
    probe = rng.standard_normal((T, k))
    loss = lambda: float((ref.route(cfg, x, w, b, sb, forced_idx=idx).weights * probe).sum())   # noqa: E731
    dl, dx, dw, db = ref.router_backward(cfg, x, w, b, sb, idx, probe)
    np.testing.assert_allclose(dx, _fd(loss, x), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dw, _fd(loss, w), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(db, _fd(loss, b), rtol=1e-6, atol=1e-8)
    # the selection-only bias carries no gradient
    np.testing.assert_allclose(_fd(loss, sb), 0.0, atol=1e-9)


def test_rms_norm_backward_finite_differences():
    rng = np.random.default_rng(11)
    z, gamma, probe = rng.standard_normal((3, 6)), rng.standard_normal(6), rng.standard_normal((3, 6))
    eps = 1e-3
    loss = lambda: float((ref.rms_norm(z, eps, gamma) * probe).sum())   # noqa: E731
    dz, dgamma = ref.rms_norm_backward(z, probe, eps, gamma)
    np.testing.assert_allclose(dz, _fd(loss, z), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dgamma, _fd(loss, gamma), rtol=1e-6, atol=1e-8)


def test_rms_norm_backward_scale_invariance():
    """Without eps the norm ignores the row's scale, so its input gradient is orthogonal to the row."""
    rng = np.random.default_rng(12)
    z, dn = rng.standard_normal((5, 16)), rng.standard_normal((5, 16))
    dz, _ = ref.rms_norm_backward(z, dn, 0.0)
    np.testing.assert_allclose((dz * z).sum(axis=1), 0.0, atol=1e-12)
    # gamma = 1 and a constant row c: r = 1/|c|, dz = (dn - mean(dn)) / |c|
    c = -2.5
    zc = np.full((1, 8), c)
    dz_c, dg_c = ref.rms_norm_backward(zc, dn[:1, :8], 0.0)
    np.testing.assert_allclose(dz_c, (dn[:1, :8] - dn[:1, :8].mean()) / abs(c), rtol=1e-13)
    np.testing.assert_allclose(dg_c, dn[0, :8] * np.sign(c), rtol=1e-13)


def test_latent_projection_backward_finite_differences():
    rng = np.random.default_rng(13)
    T, D, L = 3, 5, 4
    for norm in (1, 0):
        cfg = ref.OracleConfig(d_model=D, num_experts=2, top_k=1, hidden_size=2, gating=0, latent_dim=L,
                               up_proj_norm=norm, rms_eps=1e-3)
        z, w_up, gamma = rng.standard_normal((T, L)), rng.standard_normal((D, L)), rng.standard_normal(L)
        probe = rng.standard_normal((T, D))
        loss = lambda: float((ref.restore_routed_output(cfg, z, w_up, gamma) * probe).sum())   # noqa: E731
        dz, dw_up, dgamma = ref.restore_routed_output_backward(cfg, z, w_up, probe, gamma)
        np.testing.assert_allclose(dz, _fd(loss, z), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(dw_up, _fd(loss, w_up), rtol=1e-6, atol=1e-8)
        if norm:
            np.testing.assert_allclose(dgamma, _fd(loss, gamma), rtol=1e-6, atol=1e-8)
        else:
            assert dgamma is None
    x, w_down, probe = rng.standard_normal((T, D)), rng.standard_normal((L, D)), rng.standard_normal((T, L))
    cfg = ref.OracleConfig(d_model=D, num_experts=2, top_k=1, hidden_size=2, gating=0, latent_dim=L)
    loss = lambda: float((ref.prepare_routed_input(cfg, x, w_down) * probe).sum())   # noqa: E731
    dx, dw_down = ref.prepare_routed_input_backward(x, w_down, probe)
    np.testing.assert_allclose(dx, _fd(loss, x), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dw_down, _fd(loss, w_down), rtol=1e-6, atol=1e-8)
