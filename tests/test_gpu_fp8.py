"""GPU parity of the rowwise FP8 experts (page "Как устроен Olmo-core 3: обучение больших
MoE-моделей", §"Rowwise FP8 и MXFP8") against the float64 oracle's FP8 path: the
quantiser's codes and scales bit-exact, the layer within the layer bar."""
import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from tests.oracle_bridge import (assert_close_fp8_layer, assert_close_layer, assert_close_relative, check_topk, f64,
                                 fp8_ambiguous_tokens, oracle_config, oracle_weights)
from tests.test_gpu_parity import DESIGNED_COUNTS, designed_routing
from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WorkloadSpec, generate

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,scale", [(1000, 256, 1.0), (77, 2048, 30.0), (5, 64, 1e-3)])
def test_quantizer_bit_exact(rows, cols, scale):
    g = np.random.default_rng(rows + cols)
    x = torch.from_numpy((g.standard_normal((rows, cols)) * scale).astype(np.float32)).to(torch.bfloat16)
    x[min(3, rows - 1)] = 0.0
    codes, scales = native.moe_quantize_rowwise_fp8(x.cuda())
    assert native.moe_get_status() == 0
    want_q, want_s = ref.quantize_rowwise_e4m3(f64(x))
    np.testing.assert_array_equal(scales.cpu().numpy(), want_s)
    got_q = codes.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(got_q, want_q)


CASES = {
    "olmoe_like_small": WorkloadSpec("olmoe_like_small", T=600, d_model=512, num_experts=8, top_k=2, hidden_size=256,
                                     gating="topk_softmax", expert_fp8=True, seed=71),
    "pair_tiles_fp8": WorkloadSpec("pair_tiles_fp8", T=2000, d_model=512, num_experts=4, top_k=2, hidden_size=320,
                                   gating="sigmoid", normalize_expert_weights=1.0, expert_fp8=True, seed=72),
    "latent_fp8": WorkloadSpec("latent_fp8", T=400, d_model=768, num_experts=16, top_k=4, hidden_size=192,
                               latent_dim=256, gating="sigmoid", skew=True, expert_fp8=True, seed=73),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_layer_forward(name):
    spec = CASES[name]
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp).quantize_experts_fp8()
    ws = native.workspace(cfg, spec.T)
    out = native.moe_layer_forward(cfg, wts, inp["x"].cuda(), ws)
    assert native.moe_get_status() == 0
    inter = native.layer_intermediates(cfg, spec.T, ws)
    oc, ow = oracle_config(spec), oracle_weights(spec, inp)
    r = ref.route(oc, f64(inp["x"]), ow.w_router, ow.b_router, ow.score_bias)
    gi = inter["idx"].cpu().numpy().astype(np.int64)
    mism = check_topk(gi, r.keys, r.idx, spec.top_k)
    forced = r.idx.copy()
    forced[mism] = gi[mism]
    want = ref.layer_forward_fp8(oc, f64(inp["x"]), ow, forced_idx=forced)
    got = out.double().cpu().numpy()
    amb = fp8_ambiguous_tokens(oc, ow, f64(inp["x"]), forced)
    assert_close_fp8_layer(got, want, amb, "fp8 layer output", latent=bool(spec.latent_dim))
    # and the FP8 layer stays close to the bf16 one (e4m3 keeps 3 mantissa bits)
    dense = ref.layer_forward(oc, f64(inp["x"]), ow, forced_idx=forced).out
    assert np.linalg.norm(got - dense) / np.linalg.norm(dense) < 0.1


def test_fp8_grouped_swiglu_designed_counts():
    # every kind of group on the CTA-pair path: empty, tail only, whole tiles only, whole tiles + tail
    spec = WorkloadSpec("designed_counts_fp8", T=sum(DESIGNED_COUNTS), d_model=256,
                        num_experts=len(DESIGNED_COUNTS), top_k=1, hidden_size=192, gating="softmax",
                        expert_fp8=True, seed=74)
    assert spec.rows >= 384 * spec.num_experts
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp).quantize_experts_fp8()
    ws = native.workspace(cfg, spec.T)
    counts, offsets, gather, scatter = native.moe_permute(cfg, designed_routing(DESIGNED_COUNTS, 7), ws)
    xr = torch.from_numpy(np.random.default_rng(8).standard_normal((spec.T, spec.d_model), dtype=np.float32)).to(
        torch.bfloat16)
    y = native.moe_grouped_swiglu(cfg, wts, xr.cuda(), gather, offsets, ws)
    assert native.moe_get_status() == 0
    perm = ref.Permutation(counts.cpu().numpy(), offsets.cpu().numpy(), gather.cpu().numpy(), scatter.cpu().numpy())
    want = ref.expert_outputs_fp8(oracle_config(spec), f64(xr), perm, oracle_weights(spec, inp).expert)
    assert_close_layer(y.double().cpu().numpy(), want, "fp8 grouped swiglu, designed counts")


def test_fp8_preact():
    """e4m3 experts keep the scaled e4m3 products as pre-activations: u = x_q W_up,q and
    g = x_q W_gate,q with rowwise-dequantised operands (the quantiser is bit-exact, so only the
    accumulation order differs)."""
    spec = CASES["pair_tiles_fp8"]
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp).quantize_experts_fp8()
    ws = native.workspace(cfg, spec.T)
    x = inp["x"].cuda()
    _, idx, _ = native.moe_router(cfg, wts, x, ws)
    counts, offsets, gather, scatter = native.moe_permute(cfg, idx, ws)
    y = native.moe_grouped_swiglu(cfg, wts, x, gather, offsets, ws)
    y2, pre = native.moe_grouped_swiglu_preact(cfg, wts, x, gather, offsets, ws)
    assert native.moe_get_status() == 0
    assert torch.equal(y, y2)
    ow = oracle_weights(spec, inp)
    xq, xs = ref.quantize_rowwise_e4m3(f64(inp["x"]))
    xd = xq * xs.astype(np.float64)[:, None]
    pre = pre.double().cpu().numpy()
    off, gat = offsets.cpu().numpy(), gather.cpu().numpy()
    for e in range(spec.num_experts):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        wu, wg, _ = ref.quantize_expert_fp8(*ow.expert(e))
        rows = xd[gat[lo:hi]]
        want = np.concatenate([rows @ wu.T, rows @ wg.T], axis=1)
        assert_close_relative(pre[lo:hi], want, f"fp8 preact[{e}]")
