"""Pins of the oracle's router: gating, selection, top-k, weights, normalisation and scaling.

Page: "Как устроен Olmo-core 3: обучение больших MoE-моделей", section "Маршрутизация: как роутер выбирает
экспертов" (gating, score_bias, max for k = 1, normalisation, scalings) and
"Разрешение равенства логитов и квантизация" (lower index wins ties).
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special as sps

from oracle import moe_ref as ref


def rng(seed=0):
    return np.random.default_rng(seed)


def test_softmax_scores_match_library():
    lg = rng(1).standard_normal((7, 11)) * 3
    np.testing.assert_allclose(ref.gate_scores(lg, ref.GATING_SOFTMAX), sps.softmax(lg, axis=1), rtol=1e-13)
    np.testing.assert_allclose(ref.gate_scores(lg, ref.GATING_TOPK_SOFTMAX), sps.softmax(lg, axis=1), rtol=1e-13)
    np.testing.assert_allclose(ref.gate_scores(lg, ref.GATING_SOFTMAX).sum(1), 1.0, rtol=1e-14)


def test_sigmoid_scores_match_library_plus_epsilon():
    lg = rng(2).standard_normal((5, 9)) * 4
    eps = 1e-6
    np.testing.assert_allclose(ref.gate_scores(lg, ref.GATING_SIGMOID, eps), sps.expit(lg) + eps, rtol=1e-13)
    # the epsilon is the guard for all-very-negative logits: scores become exactly eps
    very_neg = np.full((1, 4), -700.0)
    np.testing.assert_allclose(ref.gate_scores(very_neg, ref.GATING_SIGMOID, eps), eps, rtol=1e-12)


def _brute_topk(keys_row, k):
    """All C(E, k) subsets: maximum key sum; among equal sums the smallest sorted index tuple."""
    best, best_sum = None, -math.inf
    for sub in itertools.combinations(range(len(keys_row)), k):
        s = sum(keys_row[i] for i in sub)
        if s > best_sum + 1e-12:
            best, best_sum = sub, s
    return best


@pytest.mark.parametrize("E,k", [(2, 1), (4, 2), (5, 3), (8, 2), (8, 3), (6, 6)])
def test_topk_equals_brute_force(E, k):
    keys = rng(E * 10 + k).standard_normal((16, E))
    got = ref.top_k(keys, k)
    for t in range(16):
        assert tuple(sorted(got[t])) == _brute_topk(keys[t], k)
        # descending order of the chosen keys
        assert all(keys[t, got[t, j]] > keys[t, got[t, j + 1]] for j in range(k - 1))


@pytest.mark.parametrize("E,k", [(4, 2), (6, 3), (8, 2), (8, 3)])
def test_topk_ties_lower_index_first(E, k):
    # small integer keys produce many exact ties
    keys = rng(E + 100 * k).integers(0, 3, size=(16, E)).astype(np.float64)
    got = ref.top_k(keys, k)
    for t in range(16):
        assert tuple(sorted(got[t])) == _brute_topk(keys[t], k)
        seq = [(-keys[t, e], e) for e in got[t]]
        assert seq == sorted(seq)


def test_top1_is_argmax_first_occurrence():
    keys = rng(3).integers(0, 4, size=(64, 7)).astype(np.float64)
    np.testing.assert_array_equal(ref.top_k(keys, 1)[:, 0], np.argmax(keys, axis=1))


def _cfg(**kw):
    base = dict(d_model=4, num_experts=4, top_k=2, hidden_size=4)
    base.update(kw)
    return ref.OracleConfig(**base)


def test_topk_softmax_selects_on_biased_logits_and_weights_on_selected_logits():
    # logits 0,1,2,3 (identity router on x = logits); the bias lifts expert 0 into the selection
    logits_row = np.array([[0.0, 1.0, 2.0, 3.0]])
    cfg = _cfg(gating=ref.GATING_TOPK_SOFTMAX, has_score_bias=True)
    r = ref.route(cfg, logits_row, np.eye(4), score_bias=np.array([5.0, 0.0, 0.0, 0.0]))
    np.testing.assert_array_equal(r.idx, [[0, 3]])
    # softmax over the two selected logits (0 and 3), not over all four, and not biased
    np.testing.assert_allclose(r.weights, [[1 / (1 + math.e ** 3), math.e ** 3 / (1 + math.e ** 3)]], rtol=1e-14)
    # a bias of 0.5 does not lift expert 0 when selection is on logits, but it
    # does when selection is on softmax scores (plain softmax gating):
    r2 = ref.route(cfg, logits_row, np.eye(4), score_bias=np.array([0.5, 0.0, 0.0, 0.0]))
    np.testing.assert_array_equal(r2.idx, [[3, 2]])
    r3 = ref.route(_cfg(gating=ref.GATING_SOFTMAX, has_score_bias=True), logits_row, np.eye(4),
                   score_bias=np.array([0.5, 0.0, 0.0, 0.0]))
    np.testing.assert_array_equal(r3.idx, [[3, 0]])


def test_sigmoid_bias_for_selection_only():
    logits = np.array([[0.1, 0.2, 0.3, 0.4]])
    eps = 1e-6
    cfg = _cfg(gating=ref.GATING_SIGMOID, sigmoid_stability_epsilon=eps, has_score_bias=True)
    bias = np.array([1.0, 0.0, 0.0, -1.0])
    r = ref.route(cfg, logits, np.eye(4), score_bias=bias)
    # keys: expit + eps + bias -> expert 0 first, expert 3 dropped
    np.testing.assert_array_equal(r.idx, [[0, 2]])
    np.testing.assert_allclose(r.weights, sps.expit(logits[:, [0, 2]]) + eps, rtol=1e-14)


def test_softmax_weights_are_gathered_full_softmax():
    lg = rng(5).standard_normal((6, 5))
    cfg = _cfg(num_experts=5, top_k=2, gating=ref.GATING_SOFTMAX)
    r = ref.route(cfg, lg, np.eye(5))
    full = sps.softmax(lg, axis=1)
    np.testing.assert_allclose(r.weights, np.take_along_axis(full, r.idx, 1), rtol=1e-13)
    assert (r.weights.sum(1) < 1).all()


def test_router_logits_and_router_bias():
    x = rng(6).standard_normal((3, 8))
    w = rng(7).standard_normal((5, 8))
    b = rng(8).standard_normal(5)
    cfg = _cfg(d_model=8, num_experts=5, top_k=1, router_bias=True)
    r = ref.route(cfg, x, w, b_router=b)
    np.testing.assert_allclose(r.logits, np.einsum("td,ed->te", x, w) + b, rtol=1e-12)
    # with router_bias off the given bias is ignored
    r0 = ref.route(_cfg(d_model=8, num_experts=5, top_k=1), x, w, b_router=b)
    np.testing.assert_allclose(r0.logits, np.einsum("td,ed->te", x, w), rtol=1e-12)


@pytest.mark.parametrize("gating", [ref.GATING_SOFTMAX, ref.GATING_SIGMOID, ref.GATING_TOPK_SOFTMAX])
def test_normalisation_and_scalings(gating):
    lg = rng(9).standard_normal((10, 8))
    k = 3
    base = dict(num_experts=8, top_k=k, gating=gating)
    r1 = ref.route(_cfg(normalize_expert_weights=1.0, **base), lg, np.eye(8))
    np.testing.assert_allclose(r1.weights.sum(1), 1.0, rtol=1e-13)
    r2 = ref.route(_cfg(normalize_expert_weights=2.0, **base), lg, np.eye(8))
    np.testing.assert_allclose(np.linalg.norm(r2.weights, axis=1), 1.0, rtol=1e-13)
    rr = ref.route(_cfg(normalize_expert_weights=1.0, restore_weight_scale=True, **base), lg, np.eye(8))
    np.testing.assert_allclose(rr.weights.sum(1), k, rtol=1e-13)
    rs = ref.route(_cfg(normalize_expert_weights=1.0, expert_weight_scale=2.5, **base), lg, np.eye(8))
    np.testing.assert_allclose(rs.weights.sum(1), 2.5, rtol=1e-13)
    # original_top_k = 12 with top_k = 3: x (12/3) ** 0.5 = x 2
    ro = ref.route(_cfg(normalize_expert_weights=1.0, original_top_k=12, **base), lg, np.eye(8))
    np.testing.assert_allclose(ro.weights.sum(1), 2.0, rtol=1e-13)
    rall = ref.route(_cfg(normalize_expert_weights=1.0, restore_weight_scale=True, expert_weight_scale=0.5,
                          original_top_k=12, **base), lg, np.eye(8))
    np.testing.assert_allclose(rall.weights.sum(1), k * 0.5 * 2.0, rtol=1e-13)
    # unnormalised weights keep their proportions
    r0 = ref.route(_cfg(**base), lg, np.eye(8))
    np.testing.assert_allclose(r1.weights, r0.weights / r0.weights.sum(1, keepdims=True), rtol=1e-13)


def test_forced_indices_keep_oracle_weights():
    lg = rng(10).standard_normal((4, 6))
    cfg = _cfg(num_experts=6, top_k=2, gating=ref.GATING_SIGMOID)
    forced = np.array([[5, 0], [1, 2], [3, 4], [0, 1]])
    r = ref.route(cfg, lg, np.eye(6), forced_idx=forced)
    np.testing.assert_array_equal(r.idx, forced)
    np.testing.assert_allclose(r.weights, np.take_along_axis(sps.expit(lg), forced, 1), rtol=1e-14)
