"""Pins of the oracle's permutation against library sorting and the counting-sort definition.

Page: "Как устроен Olmo-core 3: обучение больших MoE-моделей", section
"Пересылка токенов между экспертами" (indices sorted, bins = cumulative sum
of tokens per expert, scatter back by the saved indices), and section
"Балансировка нагрузки и вспомогательные штрафы" (the per-expert histogram).
"""
import numpy as np
import pytest

from oracle import moe_ref as ref


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (5, 2, 3), (64, 8, 16), (33, 3, 50), (200, 4, 7)])
def test_permutation_matches_stable_argsort(T, k, E):
    idx = np.random.default_rng(T * E + k).integers(0, E, size=(T, k))
    p = ref.permute(idx, E)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(p.counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(p.offsets, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    order = np.argsort(flat, kind="stable")          # library stable sort
    np.testing.assert_array_equal(p.gather_token, order // k)
    inv = np.empty_like(order)
    inv[order] = np.arange(T * k)
    np.testing.assert_array_equal(p.scatter_pos, inv)


def test_permutation_properties_with_empty_experts():
    T, k, E = 40, 3, 20
    idx = np.random.default_rng(3).integers(0, 5, size=(T, k)) * 4   # only experts 0,4,8,12,16
    p = ref.permute(idx, E)
    assert p.counts.sum() == T * k
    assert (p.counts[[e for e in range(E) if e % 4]] == 0).all()
    flat = idx.reshape(-1)
    # row p of the permuted order belongs to the bin of its expert
    for e in range(E):
        lo, hi = p.offsets[e], p.offsets[e + 1]
        rows = np.arange(lo, hi)
        src = np.nonzero(flat == e)[0]
        np.testing.assert_array_equal(p.scatter_pos[src], rows)    # ascending flat order inside the bin
        np.testing.assert_array_equal(p.gather_token[rows], src // k)
    # scatter then gather is the identity on assignments
    np.testing.assert_array_equal(p.gather_token[p.scatter_pos], np.arange(T * k) // k)


def test_permutation_empty_batch():
    p = ref.permute(np.zeros((0, 4), np.int64), 6)
    assert p.counts.tolist() == [0] * 6 and p.offsets.tolist() == [0] * 7
    assert p.gather_token.size == 0 and p.scatter_pos.size == 0
