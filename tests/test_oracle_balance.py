"""Pins of the oracle's load-balancing counters, section "Счётчики и bias-корректировка" of the
page "Как устроен Olmo-core 3: обучение больших MoE-моделей": accumulation, the max / mean
imbalance metric and the sign-based score-bias correction, on hand-computed cases."""
import math

import numpy as np

from oracle import moe_ref as ref


def test_accumulate_counts():
    acc = ref.accumulate_counts(np.array([1, 2, 3]), np.array([4, 0, 1]))
    np.testing.assert_array_equal(acc, [5, 2, 4])
    assert acc.dtype == np.int64


def test_load_imbalance_hand_values():
    assert ref.load_imbalance(np.array([3, 1, 2, 2])) == 1.5     # max 3 / mean 2
    assert ref.load_imbalance(np.array([5, 5, 5])) == 1.0        # balanced
    assert ref.load_imbalance(np.array([8, 0, 0, 0])) == 4.0     # all on one expert: E
    assert math.isnan(ref.load_imbalance(np.array([0, 0])))


def test_score_bias_update_hand_values():
    bias = np.array([0.5, -0.25, 0.0, 1.0])
    accum = np.array([3, 1, 2, 2])                               # ideal = 2
    new, zeroed = ref.score_bias_update(bias, accum, 0.125)
    # above the mean: -gamma; below: +gamma; equal: unchanged
    np.testing.assert_array_equal(new, [0.375, -0.125, 0.0, 1.0])
    np.testing.assert_array_equal(zeroed, [0, 0, 0, 0])


def test_score_bias_update_non_integer_ideal_and_balance_direction():
    accum = np.array([10, 0, 1])                                 # ideal 11/3
    new, _ = ref.score_bias_update(np.zeros(3), accum, 1.0)
    np.testing.assert_array_equal(new, [-1.0, 1.0, 1.0])
    # repeated corrections push an over-loaded expert's bias down monotonically
    b = np.zeros(3)
    for _ in range(4):
        b, _ = ref.score_bias_update(b, accum, 0.5)
    np.testing.assert_array_equal(b, [-2.0, 2.0, 2.0])
