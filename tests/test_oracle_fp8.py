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


def test_mx_quantiser_closed_forms():
    """MX blocks: the scale exponent is floor(log2 amax) - 8 + 127, codes = e4m3(v / 2^(e-127)); a block
    whose values are e4m3 values times a power of two comes back exactly, an all-zero block has e = 0."""
    g = np.random.default_rng(3)
    codes = g.choice(ref._E4M3[ref._E4M3 <= 448], size=(4, 64)) * g.choice([-1.0, 1.0], size=(4, 64))
    codes[:, 0] = 448.0                                   # block amax 448 = 1.75 * 2^8: floor(log2) = 8
    codes[:, 32] = -448.0
    x = codes * 2.0 ** np.array([-20, -3, 0, 7])[:, None]
    q, e = ref.quantize_mx_e4m3(x)
    np.testing.assert_array_equal(e, np.array([[107, 107], [124, 124], [127, 127], [134, 134]]))
    np.testing.assert_array_equal(ref.dequantize_mx(q, e), x)
    z = np.zeros((2, 32))
    qz, ez = ref.quantize_mx_e4m3(z)
    assert (qz == 0).all() and (ez == 0).all()


def test_mx_quantiser_saturates_and_bounds_the_error():
    """amax / X lies in [256, 512): values above 448 saturate; every other value is within half an
    e4m3 step of v / X (relative 2^-4), and the scale is a power of two chosen per 32-value block."""
    g = np.random.default_rng(4)
    x = g.standard_normal((64, 256)) * np.exp(g.uniform(-8, 8, size=(64, 1)))
    q, e = ref.quantize_mx_e4m3(x)
    d = ref.dequantize_mx(q, e)
    blocks = x.reshape(64, 8, 32)
    scale = 2.0 ** (e - 127)
    amax = np.abs(blocks).max(axis=2)
    assert ((amax / scale >= 256) & (amax / scale < 512)).all()
    v = blocks / scale[:, :, None]
    sat = np.abs(v) > 448
    assert (np.abs(q.reshape(64, 8, 32))[sat] == 448).all()
    err = np.abs(d.reshape(64, 8, 32) - blocks)[~sat] / np.maximum(np.abs(blocks[~sat]), 2.0 ** -6 * scale.repeat(32).reshape(64, 8, 32)[~sat])
    assert err.max() <= 2.0 ** -4 + 1e-12
    # block-wise: each 32-wide block of a row has its own exponent
    x2 = np.concatenate([np.full((1, 32), 1.0), np.full((1, 32), 1000.0)], axis=1)
    _, e2 = ref.quantize_mx_e4m3(x2)
    np.testing.assert_array_equal(e2, [[0 - 8 + 127, 9 - 8 + 127]])


def test_mx_experts_reduce_to_the_exact_experts_on_representable_inputs():
    """When x, the weights and H are all MX-representable, the MXFP8 experts equal the exact ones
    (H rounded to bf16 and re-quantised in between)."""
    cfg = ref.OracleConfig(d_model=64, num_experts=2, top_k=1, hidden_size=32)
    g = np.random.default_rng(5)
    pick = lambda shape: g.choice([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0], size=shape)   # noqa: E731
    x = pick((6, 64))
    w = [(pick((32, 64)) / 8, pick((32, 64)) / 8, pick((64, 32)) / 8) for _ in range(2)]
    perm = ref.permute(np.array([[0], [1], [0], [1], [1], [0]]), 2)
    got = ref.expert_outputs_mxfp8(cfg, x, perm, lambda e: w[e])
    h_exact = {}
    want = np.zeros_like(got)
    for e in range(2):
        lo, hi = int(perm.offsets[e]), int(perm.offsets[e + 1])
        rows = x[perm.gather_token[lo:hi]]
        h = ref.round_bf16(ref.silu(rows @ w[e][1].T) * (rows @ w[e][0].T))
        want[lo:hi] = ref.dequantize_mx(*ref.quantize_mx_e4m3(h)) @ w[e][2].T
        h_exact[e] = h
    np.testing.assert_allclose(got, want, rtol=0, atol=0)


def test_mx_experts_hand_computed_h_rounding():
    """One token through one expert, every operand MX-representable and every value worked out by
    hand.  x = (1, 1, 0, ...); gate rows 0, 1 give g = 32 + 32 = 64, where silu(64) = 64 exactly
    in float64 (e^-64 is below half an ulp); up rows give u0 = 1 + 0.0625 and u1 = 2.  So
    h = (68, 128, 0, ...), exact in bf16.  H's first block has amax 128 = 2^7, so its scale is
    2^(7 - 8) = 1/2 and 68 / (1/2) = 136 lies halfway between the e4m3 neighbours 128 and 144: the
    tie goes to the even code 128, and h0 comes back as 64.  W_out copies H's first two columns, so
    the output is (64, 128, 0, ...) where the unquantised expert gives (68, 128, 0, ...)."""
    D, h = 64, 32
    cfg = ref.OracleConfig(d_model=D, num_experts=1, top_k=1, hidden_size=h)
    x = np.zeros((1, D))
    x[0, :2] = 1.0
    w_up, w_gate, w_out = np.zeros((h, D)), np.zeros((h, D)), np.zeros((D, h))
    w_up[0, :2] = [1.0, 0.0625]
    w_up[1, 0] = 2.0
    w_gate[0, :2] = w_gate[1, :2] = 32.0
    w_out[0, 0] = w_out[1, 1] = 1.0
    perm = ref.permute(np.array([[0]]), 1)
    got = ref.expert_outputs_mxfp8(cfg, x, perm, lambda e: (w_up, w_gate, w_out))
    want = np.zeros((1, D))
    want[0, :2] = [64.0, 128.0]
    np.testing.assert_array_equal(got, want)
    exact = ref.expert_outputs(cfg, x, perm, lambda e: (w_up, w_gate, w_out))
    assert exact[0, 0] == 68.0 and exact[0, 1] == 128.0



# ---------------------------------------------------------------------------
# Rowwise FP8 experts.  Every value below is worked out by hand.  A row scale is amax / 448 in
# float32; it is exact when amax = 7 * 2^m (448 = 7 * 2^6), so the rows are built that way.
# ---------------------------------------------------------------------------

def _fp8_hand_expert(D=64, h=32):
    """x = (7, 4, 0, ...): scale 7 / 448 = 2^-6, codes (448, 256).  Gate rows 0, 1 = (7, 3.75):
    scale 2^-6, codes (448, 240), g = 49 + 15 = 64, and silu(64) = 64 exactly in float64 (e^-64 is
    below half an ulp of 1).  Up row 0 = (7/32, -15/128): scale 2^-11, codes (448, -240),
    u0 = 49/32 - 15/32 = 17/16.  Up row 1 = (7/8, 7/32): scale 2^-9, codes (448, 112), u1 = 7.
    So H = (68, 448, 0, ...), exact in bf16.  H's row amax 448 gives the row scale 1, and 68 lies
    halfway between the e4m3 neighbours 64 and 72: the tie goes to the even code, 64.  W_out rows
    0, 1 hold 7/8 in columns 0, 1 (scale 2^-9, code 448), so y = 7/8 * (64, 448) = (56, 392),
    where the unquantised expert gives 7/8 * (68, 448) = (59.5, 392)."""
    w_up, w_gate, w_out = np.zeros((h, D)), np.zeros((h, D)), np.zeros((D, h))
    w_gate[0, :2] = w_gate[1, :2] = [7.0, 3.75]
    w_up[0, :2] = [7.0 / 32, -15.0 / 128]
    w_up[1, :2] = [7.0 / 8, 7.0 / 32]
    w_out[0, 0] = w_out[1, 1] = 7.0 / 8
    return w_up, w_gate, w_out


def test_rowwise_expert_weights_round_trip_when_representable():
    """quantize_expert_fp8 returns rows whose amax is 7 * 2^m and whose other entries are e4m3
    codes times that row's scale unchanged; the scale belongs to the row, not the column."""
    g = np.random.default_rng(6)
    codes = ref._E4M3[ref._E4M3 <= 448]

    def rows(n, cols):
        c = g.choice(codes, size=(n, cols)) * g.choice([-1.0, 1.0], size=(n, cols))
        c[np.arange(n), g.integers(0, cols, n)] = 448.0 * g.choice([-1.0, 1.0], size=n)   # each row's amax code
        return c * 2.0 ** g.integers(-14, 2, size=(n, 1)) / 64.0                          # scale 2^m / 64
    mats = (rows(16, 48), rows(16, 48), rows(48, 16))
    for got, want in zip(ref.quantize_expert_fp8(*mats), mats):
        np.testing.assert_array_equal(got, want)
    _, s = ref.quantize_rowwise_e4m3(mats[0])
    np.testing.assert_array_equal(s, np.abs(mats[0]).max(axis=1) / 448.0)


def test_fp8_experts_hand_computed_h_tie():
    cfg = ref.OracleConfig(d_model=64, num_experts=1, top_k=1, hidden_size=32)
    x = np.zeros((1, 64))
    x[0, :2] = [7.0, 4.0]
    w = _fp8_hand_expert()
    perm = ref.permute(np.array([[0]]), 1)
    got = ref.expert_outputs_fp8(cfg, x, perm, lambda e: w)
    want = np.zeros((1, 64))
    want[0, :2] = [56.0, 392.0]
    np.testing.assert_array_equal(got, want)
    exact = ref.expert_outputs(cfg, x, perm, lambda e: w)
    assert exact[0, 0] == 59.5 and exact[0, 1] == 392.0


def test_fp8_latent_layer_hand_computed():
    """The latent FP8 layer quantises the experts' bf16 input.  x = (1, 1, 0, ...) and W_down rows
    (7, 2^-6, 0, ...), (4, 0, ...) give x_routed = (7 + 2^-6, 4): 7 + 2^-6 lies halfway between the
    bf16 neighbours 7 and 7 + 2^-5 and goes to the even one, 7.  From there the expert above gives
    (56, 392).  One expert with softmax gating has weight 1; with the norm off and W_up the
    identity the layer output is z itself."""
    D = L = 64
    cfg = ref.OracleConfig(d_model=D, num_experts=1, top_k=1, hidden_size=32, latent_dim=L, up_proj_norm=False)
    x = np.zeros((1, D))
    x[0, :2] = 1.0
    w_down = np.zeros((L, D))
    w_down[0, :2] = [7.0, 2.0 ** -6]
    w_down[1, 0] = 4.0
    w = _fp8_hand_expert(D=L)
    wts = ref.OracleWeights(w_router=np.zeros((1, D)), expert=lambda e: w, w_down_latent=w_down,
                            w_up_latent=np.eye(D, L))
    got = ref.layer_forward_fp8(cfg, x, wts)
    want = np.zeros((1, D))
    want[0, :2] = [56.0, 392.0]
    np.testing.assert_array_equal(got, want)


def test_mx_latent_layer_hand_computed():
    """The latent MXFP8 layer quantises the experts' bf16 input, worked out by hand.  x = (1, 1, 0, ...)
    and W_down rows (1.1875, -2^-9, 0, ...), (1, 0, ...) give x_routed = (1.1875 - 2^-9, 1).  bf16
    rounds the first to 1.1875 (2^-9 is under half its step of 2^-7).  That row's block amax is
    1.1875, so its scale is 2^(0 - 8) and 1.1875 / 2^-8 = 304, halfway between the e4m3 neighbours
    288 and 320: the tie goes to the even code 320, so the expert sees x = (1.25, 1).  (Without the
    bf16 rounding, 303.5 goes to 288 and x0 = 1.125.)  Gate rows 0, 1 = (32, 32): g = 72 and
    silu(72) = 72 in float64.  Up rows (1, 1/16) and (2, 0): u = (1.3125, 2.5).  So H = (94.5, 180),
    exact in bf16; its block amax 180 gives the scale 1/2, and 189 rounds to the e4m3 code 192,
    360 to 352: H = (96, 176).  W_out copies H's first two columns; one expert with softmax gating
    has weight 1, and with the norm off and W_up the identity the output is (96, 176, 0, ...).  Every
    weight row is MX-representable (codes 256 and 16 under power-of-two scales)."""
    D = L = 64
    h = 32
    cfg = ref.OracleConfig(d_model=D, num_experts=1, top_k=1, hidden_size=h, latent_dim=L, up_proj_norm=False)
    x = np.zeros((1, D))
    x[0, :2] = 1.0
    w_down = np.zeros((L, D))
    w_down[0, :2] = [1.1875, -(2.0 ** -9)]
    w_down[1, 0] = 1.0
    w_up, w_gate, w_out = np.zeros((h, L)), np.zeros((h, L)), np.zeros((L, h))
    w_up[0, :2] = [1.0, 0.0625]
    w_up[1, 0] = 2.0
    w_gate[0, :2] = w_gate[1, :2] = 32.0
    w_out[0, 0] = w_out[1, 1] = 1.0
    wts = ref.OracleWeights(w_router=np.zeros((1, D)), expert=lambda e: (w_up, w_gate, w_out), w_down_latent=w_down,
                            w_up_latent=np.eye(D, L))
    got = ref.layer_forward_mxfp8(cfg, x, wts)
    want = np.zeros((1, D))
    want[0, :2] = [96.0, 176.0]
    np.testing.assert_array_equal(got, want)


def test_bf16_half_ulp_bound_is_the_rounding_error():
    """half_ulp_bf16 bounds |v - bf16(v)| and is reached at rounding midpoints (the parity bar's
    allowance for a bf16 output's own rounding)."""
    from tests.oracle_bridge import half_ulp_bf16
    v = np.random.default_rng(7).standard_normal(50000) * np.exp(np.random.default_rng(8).uniform(-20, 20, 50000))
    v = v.astype(np.float32).astype(np.float64)    # a GPU result is rounded to bf16 from float32
    assert (np.abs(ref.round_bf16(v) - v) <= half_ulp_bf16(v)).all()
    mid = np.array([1.0 + 2.0 ** -8, 8.0 + 2.0 ** -5, -(4.0 + 2.0 ** -6)])       # halfway between bf16 neighbours
    np.testing.assert_array_equal(np.abs(ref.round_bf16(mid) - mid), half_ulp_bf16(mid))
    np.testing.assert_array_equal(half_ulp_bf16(np.array([0.0, 1.0, 7.99, 8.0, 15.9])),
                                  [0.0, 2.0 ** -8, 2.0 ** -6, 2.0 ** -5, 2.0 ** -5])
