"""Pins of the oracle's rowwise FP8 path: e4m3 rounding against torch's float8_e4m3fn
conversion (a library routine), bf16 rounding against torch, and the quantiser's invariants."""
import numpy as np
import torch

from oracle import moe_ref as ref


def test_e4m3_rounding_matches_torch():
    g = np.random.default_rng(0)
    v = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * 50,
        g.standard_normal(5000).astype(np.float32) * 1e-3,
        ref._E4M3.astype(np.float32),                                   # every code exactly
        ((ref._E4M3[1:] + ref._E4M3[:-1]) / 2).astype(np.float32),      # every midpoint: ties to even
        np.array([448, 460, 463.9, -448, 0, -0.0, 2 ** -10, 3 * 2 ** -11], np.float32),
    ])
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(ref.round_e4m3(v.astype(np.float64)), want)


def test_bf16_rounding_matches_torch():
    v = (np.random.default_rng(1).standard_normal(20000) * 10).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ref.round_bf16(v), want)


def test_rowwise_quantiser_invariants():
    x = np.random.default_rng(2).standard_normal((50, 256)) * np.linspace(0.01, 100, 50)[:, None]
    x[7] = 0.0
    q, s = ref.quantize_rowwise_e4m3(x)
    assert s.dtype == np.float32 and s[7] == 1.0 and (q[7] == 0).all()
    assert np.abs(q).max() <= 448.0
    np.testing.assert_array_equal(np.abs(q[np.arange(50) != 7]).max(axis=1), 448.0)   # each row's max hits 448
    rel = np.abs(q * s[:, None] - x) / np.maximum(np.abs(x), 1e-30)
    assert (rel[np.abs(x) > s[:, None] * 2.0 ** -6] <= 2.0 ** -4 + 1e-6).all()         # e4m3: 3 mantissa bits


def test_fp8_ambiguity_band_flags_rows_at_a_rounding_midpoint():
    # bf16 keeps 8 significant bits: 1 + 2^-8 lies exactly halfway between 1 and 1 + 2^-7
    from tests.oracle_bridge import _amax_ambiguous
    rows = np.array([[0.5, 1.0 + 2.0 ** -8, -0.25],     # amax on a midpoint: either neighbour
                     [0.5, 1.0 + 2.0 ** -7, -0.25],     # amax exactly representable
                     [0.5, -(1.0 + 2.0 ** -8), 0.25]])  # the sign does not matter
    np.testing.assert_array_equal(_amax_ambiguous(rows, 1e-5), [True, False, True])
