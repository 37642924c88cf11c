"""Pins of the oracle's capacity mode, section "Ёмкость эксперта и переполнение" of the page
"Как устроен Olmo-core 3: обучение больших MoE-моделей": the capacity formula on hand values,
dropping at the permutation by brute force, and the no-drop limit equal to the dropless layer."""
import numpy as np

from oracle import moe_ref as ref
from tests.test_oracle_layer import _weights


def _cfg(E, k):
    return ref.OracleConfig(d_model=16, num_experts=E, top_k=k, hidden_size=8)


def test_capacity_formula_hand_values():
    assert ref.expert_capacity(_cfg(64, 8), 8192, 1.25) == 1280    # ideal 1024, x1.25
    assert ref.expert_capacity(_cfg(8, 2), 100, 1.0) == 32         # ideal 25 -> next multiple of 8
    assert ref.expert_capacity(_cfg(8, 2), 100, 0.5) == 16         # 12.5 -> 16
    assert ref.expert_capacity(_cfg(8, 2), 96, 1.0) == 24          # 24 exactly
    assert ref.expert_capacity(_cfg(8, 2), 100, 1.0, ep_degree=4) == 128


def test_dropping_keeps_the_first_assignments_of_each_expert():
    g = np.random.default_rng(0)
    T, k, E, cap = 50, 3, 5, 16
    idx = g.choice(E, size=(T, k), p=[0.5, 0.2, 0.1, 0.1, 0.1])
    p = ref.permute_with_capacity(idx, E, cap)
    flat = idx.reshape(-1)
    for e in range(E):
        mine = np.nonzero(flat == e)[0]                      # ascending flat order
        kept, dropped = mine[:cap], mine[cap:]
        np.testing.assert_array_equal(p.scatter_slot[kept], e * cap + np.arange(len(kept)))
        assert (p.scatter_slot[dropped] == -1).all()
        np.testing.assert_array_equal(p.slot_token[e * cap:e * cap + len(kept)], kept // k)
        assert (p.slot_token[e * cap + len(kept):(e + 1) * cap] == -1).all()
    np.testing.assert_array_equal(p.counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(p.kept, np.minimum(p.counts, cap))


def test_no_drop_limit_equals_dropless_layer():
    T, D, E, h, k = 24, 16, 4, 8, 2
    w, *_ = _weights(D, D, E, h, seed=31)
    x = np.random.default_rng(32).standard_normal((T, D))
    cfg = ref.OracleConfig(d_model=D, num_experts=E, top_k=k, hidden_size=h, gating=ref.GATING_SIGMOID)
    _, perm, _, _, out = ref.layer_forward_capacity(cfg, x, w, capacity_factor=8.0)
    assert (perm.scatter_slot >= 0).all()
    np.testing.assert_allclose(out, ref.layer_forward(cfg, x, w).out, rtol=1e-13, atol=1e-15)


def test_dropped_assignments_add_nothing():
    T, D, E, h, k = 40, 16, 4, 8, 2
    w, *_ = _weights(D, D, E, h, seed=33)
    x = np.random.default_rng(34).standard_normal((T, D))
    cfg = ref.OracleConfig(d_model=D, num_experts=E, top_k=k, hidden_size=h, gating=ref.GATING_SOFTMAX)
    r, perm, y, z, out = ref.layer_forward_capacity(cfg, x, w, capacity_factor=0.25)   # cap 8 of ~20
    assert (perm.scatter_slot == -1).sum() > 0
    full = ref.layer_forward(cfg, x, w, forced_idx=r.idx)
    # per token: the dense result minus the dropped experts' weighted outputs
    for t in range(T):
        want = full.z[t].copy()
        for j in range(k):
            if perm.scatter_slot[t * k + j] < 0:
                want -= r.weights[t, j] * full.y[full.perm.scatter_pos[t * k + j]]
        np.testing.assert_allclose(z[t], want, rtol=1e-12, atol=1e-12)
