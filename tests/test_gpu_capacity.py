"""GPU parity of capacity mode (page "Как устроен Olmo-core 3: обучение больших MoE-моделей",
§"Ёмкость эксперта и переполнение") against the float64 oracle: slots, drops and padding
bit-exact on the GPU's own routing; expert outputs and the layer within the layer bar; and the
no-drop limit equal, bit for bit, to the dropless layer."""
import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from tests.oracle_bridge import (assert_close_layer, capacity_factor_f32, check_topk, f64, oracle_config,
                                 oracle_weights)
from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WorkloadSpec, generate

pytestmark = pytest.mark.gpu

CASES = {
    "drops": WorkloadSpec("drops", T=600, d_model=512, num_experts=16, top_k=4, hidden_size=256, gating="sigmoid",
                          skew=True, capacity_factor=0.5, seed=41),
    "some_drops_latent": WorkloadSpec("some_drops_latent", T=500, d_model=768, num_experts=12, top_k=3,
                                      hidden_size=192, latent_dim=256, gating="softmax", skew=True,
                                      normalize_expert_weights=1.0, capacity_factor=1.0, seed=42),
    "pair_tiles_capacity": WorkloadSpec("pair_tiles_capacity", T=2000, d_model=512, num_experts=4, top_k=2,
                                        hidden_size=256, gating="topk_softmax", capacity_factor=1.25, seed=43),
}

_cache = {}


def setup(name):
    if name not in _cache:
        spec = CASES[name]
        inp = generate(spec)
        _cache[name] = (spec, inp, native.config_from_spec(spec), native.DeviceWeights.from_inputs(inp))
    return _cache[name]


@pytest.mark.parametrize("name", list(CASES))
def test_capacity_permutation_bit_exact(name):
    spec, inp, cfg, wts = setup(name)
    ws = native.workspace(cfg, spec.T)
    _, idx, _ = native.moe_router(cfg, wts, inp["x"].cuda(), ws)
    counts, offsets, gather, scatter = native.moe_permute(cfg, idx, ws)
    assert native.moe_get_status() == 0
    cap = native.moe_expert_capacity(cfg, spec.T)
    assert cap == ref.expert_capacity(oracle_config(spec), spec.T, capacity_factor_f32(spec))
    p = ref.permute_with_capacity(idx.cpu().numpy(), spec.num_experts, cap)
    np.testing.assert_array_equal(counts.cpu().numpy(), p.counts)
    np.testing.assert_array_equal(offsets.cpu().numpy(), np.arange(spec.num_experts + 1) * cap)
    np.testing.assert_array_equal(gather.cpu().numpy(), p.slot_token)
    np.testing.assert_array_equal(scatter.cpu().numpy(), p.scatter_slot)
    if name == "drops":
        assert (p.scatter_slot < 0).sum() > 0 and (p.slot_token < 0).sum() > 0   # both drops and padding


@pytest.mark.parametrize("name", list(CASES))
def test_capacity_experts_and_combine(name):
    spec, inp, cfg, wts = setup(name)
    T, Lr = spec.T, spec.routed_dim
    ws = native.workspace(cfg, T)
    _, idx, w = native.moe_router(cfg, wts, inp["x"].cuda(), ws)
    counts, offsets, gather, scatter = native.moe_permute(cfg, idx, ws)
    xr = torch.from_numpy(np.random.default_rng(spec.seed + 7).standard_normal((T, Lr), dtype=np.float32)).to(
        torch.bfloat16)
    y = native.moe_grouped_swiglu(cfg, wts, xr.cuda(), gather, offsets, ws)
    z = native.moe_combine(cfg, y, scatter, w, T)
    assert native.moe_get_status() == 0
    cap = native.moe_expert_capacity(cfg, T)
    p = ref.permute_with_capacity(idx.cpu().numpy(), spec.num_experts, cap)
    want_y = ref.expert_outputs_capacity(oracle_config(spec), f64(xr), p, oracle_weights(spec, inp).expert)
    got_y = y.double().cpu().numpy()
    assert (got_y[p.slot_token < 0] == 0).all()             # padding slots compute zero rows
    assert_close_layer(got_y, want_y, "capacity expert outputs")
    want_z = ref.combine_capacity(got_y, p.scatter_slot, w.double().cpu().numpy())
    got_z = z.double().cpu().numpy()
    assert np.all(np.abs(got_z - want_z) <= 2.0 ** -8 * np.abs(want_z) + 1e-5)


@pytest.mark.parametrize("name", list(CASES))
def test_capacity_layer_forward(name):
    spec, inp, cfg, wts = setup(name)
    T, k = spec.T, spec.top_k
    ws = native.workspace(cfg, T)
    out = native.moe_layer_forward(cfg, wts, inp["x"].cuda(), ws)
    assert native.moe_get_status() == 0
    inter = native.layer_intermediates(cfg, T, ws)
    oc, ow = oracle_config(spec), oracle_weights(spec, inp)
    r = ref.route(oc, f64(inp["x"]), ow.w_router, ow.b_router, ow.score_bias)
    gi = inter["idx"].cpu().numpy().astype(np.int64)
    mism = check_topk(gi, r.keys, r.idx, k)
    forced = r.idx.copy()
    forced[mism] = gi[mism]
    *_, want = ref.layer_forward_capacity(oc, f64(inp["x"]), ow, capacity_factor_f32(spec), forced_idx=forced)
    assert_close_layer(out.double().cpu().numpy(), want, "capacity layer output")


def test_no_drop_limit_is_the_dropless_layer_bit_for_bit():
    spec = WorkloadSpec("no_drop", T=700, d_model=512, num_experts=8, top_k=2, hidden_size=256, gating="sigmoid",
                        seed=44)
    inp = generate(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    x = inp["x"].cuda()
    dense_cfg = native.config_from_spec(spec)
    cap_cfg = native.config_from_spec(spec.with_(capacity_factor=8.0))
    a = native.moe_layer_forward(dense_cfg, wts, x, native.workspace(dense_cfg, spec.T))
    b = native.moe_layer_forward(cap_cfg, wts, x, native.workspace(cap_cfg, spec.T))
    assert native.moe_get_status() == 0
    assert torch.equal(a, b)
