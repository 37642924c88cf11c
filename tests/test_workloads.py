"""The seeded input generator: deterministic, correctly shaped, experts redrawable alone."""
import numpy as np
import torch

from token_routing_expert_gb300 import workloads as W


def test_tiny_workload_shapes_and_determinism():
    spec = W.WORKLOADS["tiny"]
    a = W.generate(spec)
    b = W.generate(spec, threads=1)
    for key in ("x", "w_router", "w_up_gate", "w_out"):
        assert a[key].dtype == torch.bfloat16
        assert torch.equal(a[key], b[key])
    assert a["x"].shape == (256, 256)
    assert a["w_up_gate"].shape == (8, 256, 256) and a["w_out"].shape == (8, 256, 128)
    assert a["b_router"] is None and a["score_bias"] is None and a["w_down"] is None
    # spread of the draws: x ~ N(0, 1), weights ~ N(0, 0.02)
    assert abs(a["x"].float().std().item() - 1.0) < 0.02
    assert abs(a["w_out"].float().std().item() - 0.02) < 0.001


def test_expert_redrawn_alone_matches_full_draw():
    spec = W.WORKLOADS["tiny"].with_(num_experts=5)
    full = W.generate(spec, threads=3)
    ug, o = W.expert_weights(spec, 3)
    assert torch.equal(full["w_up_gate"][3], ug) and torch.equal(full["w_out"][3], o)


def test_skew_bias_is_half_log_inverse_rank():
    spec = W.WORKLOADS["latent_prefill"].with_(num_experts=16)
    b = W.skew_bias(spec)
    ranks = np.rint(np.exp(-2.0 * b.astype(np.float64))).astype(int)
    assert sorted(ranks.tolist()) == list(range(1, 17))
    assert b.max() == 0.0


def test_named_workloads():
    assert set(W.WORKLOADS) == {"tiny", "olmoe", "sigmoid_wide", "latent_prefill", "latent_decode"}
    s = W.WORKLOADS["sigmoid_wide"]
    assert s.gating == "sigmoid" and s.score_bias_std == 0.01 and s.restore_weight_scale
    assert W.algorithmic_flops(W.WORKLOADS["olmoe"]) == 2 * 8192 * 2048 * 64 + 6 * 2048 * 1024 * 8192 * 8
