"""Full-size parity of the other modes bench.py times: rowwise FP8 experts
(`--fp8`), MXFP8 experts (`--mxfp8`) and the capacity-factor layer
(`--capacity-factor`), in the same launch configuration (one moe_layer_forward
with the library's own workspace).

FP8: the top-k indices on all tokens (near-tie rule), and sampled tokens'
outputs against the float64 oracle's FP8 layer run on those tokens alone (FP8
quantises per token and per weight row, so tokens stay independent).  A token
whose routed row or SwiGLU row has its bf16 amax within computation error of a
rounding midpoint may quantise that whole row with the neighbouring scale: such
tokens are found from the oracle's own values and held to rel-L2 only.  A latent
layer's quantiser input is itself computed (the down-projection), and is held to
the FP8 bar: rel-L2 1e-2 over the sample, half an e4m3 step per token.

MXFP8: as FP8, with the oracle's MXFP8 layer on the sampled tokens (the block
scales belong to one token's row or one weight row, so tokens stay independent),
held to the MXFP8 bar of the small-case tests: rel-L2 1e-2 over the sample and
half an e4m3 step per token.

Capacity: the capacity permutation over all tokens bit-exact against the
oracle's on the GPU's indices.  Which assignments drop depends on every token,
so the sampled tokens are recomputed by the oracle with the dropped
assignments' weights set to zero.
"""
import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from tests.oracle_bridge import (assert_close_fp8_layer, assert_close_layer, capacity_factor_f32, check_topk, f64,
                                 fp8_ambiguous_tokens, oracle_config, oracle_weights)
from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WORKLOADS, generate

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLE = 64


def _run(spec):
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    if spec.expert_fp8 == native.EXPERT_MXFP8:
        wts.quantize_experts_mxfp8()
    elif spec.expert_fp8:
        wts.quantize_experts_fp8()
    ws = native.workspace(cfg, spec.T)
    out = native.moe_layer_forward(cfg, wts, inp["x"].cuda(), ws)
    assert native.moe_get_status() == 0
    inter = {k: v.cpu() for k, v in native.layer_intermediates(cfg, spec.T, ws).items()
             if k in ("idx", "counts", "offsets", "gather_idx", "scatter_idx")}
    return inp, cfg, out.double().cpu().numpy(), inter


@pytest.mark.parametrize("name", ["olmoe", "latent_prefill"])
def test_full_size_fp8(name):
    spec = WORKLOADS[name].with_(expert_fp8=True)
    inp, cfg, out, inter = _run(spec)
    gi = inter["idx"].numpy().astype(np.int64)
    oc, ow = oracle_config(spec), oracle_weights(spec, inp)
    r = ref.route(oc, f64(inp["x"]), ow.w_router, ow.b_router, ow.score_bias)
    mism = check_topk(gi, r.keys, r.idx, spec.top_k)
    sample = np.sort(np.random.default_rng(4321).choice(spec.T, size=SAMPLE, replace=False))
    forced = r.idx[sample].copy()
    forced[mism[sample]] = gi[sample][mism[sample]]
    xs = f64(inp["x"][torch.from_numpy(sample)])
    want = ref.layer_forward_fp8(oc, xs, ow, forced_idx=forced)
    amb = fp8_ambiguous_tokens(oc, ow, xs, forced)
    assert_close_fp8_layer(out[sample], want, amb, f"{name} fp8 sampled layer output",
                           latent=bool(spec.latent_dim))


@pytest.mark.parametrize("name", ["olmoe", "latent_prefill"])
def test_full_size_mxfp8(name):
    from tests.test_gpu_mxfp8 import assert_close_mx
    spec = WORKLOADS[name].with_(expert_fp8=native.EXPERT_MXFP8)
    inp, cfg, out, inter = _run(spec)
    gi = inter["idx"].numpy().astype(np.int64)
    oc, ow = oracle_config(spec), oracle_weights(spec, inp)
    r = ref.route(oc, f64(inp["x"]), ow.w_router, ow.b_router, ow.score_bias)
    mism = check_topk(gi, r.keys, r.idx, spec.top_k)
    sample = np.sort(np.random.default_rng(4322).choice(spec.T, size=SAMPLE, replace=False))
    forced = r.idx[sample].copy()
    forced[mism[sample]] = gi[sample][mism[sample]]
    want = ref.layer_forward_mxfp8(oc, f64(inp["x"][torch.from_numpy(sample)]), ow, forced_idx=forced)
    assert_close_mx(out[sample], want, f"{name} mxfp8 sampled layer output")


def test_full_size_capacity():
    spec = WORKLOADS["olmoe"].with_(capacity_factor=1.0)   # capacity 1024: the fullest experts overflow
    inp, cfg, out, inter = _run(spec)
    E, k, T = spec.num_experts, spec.top_k, spec.T
    gi = inter["idx"].numpy().astype(np.int64)
    oc, ow = oracle_config(spec), oracle_weights(spec, inp)
    r = ref.route(oc, f64(inp["x"]), ow.w_router, ow.b_router, ow.score_bias)
    mism = check_topk(gi, r.keys, r.idx, k)
    cap = ref.expert_capacity(oc, T, capacity_factor_f32(spec))
    assert native.moe_expert_capacity(cfg, T) == cap
    perm = ref.permute_with_capacity(gi, E, cap)
    np.testing.assert_array_equal(inter["counts"].numpy(), perm.counts)
    np.testing.assert_array_equal(inter["gather_idx"].numpy(), perm.slot_token)
    np.testing.assert_array_equal(inter["scatter_idx"].numpy(), perm.scatter_slot)
    assert (perm.scatter_slot < 0).any() and (perm.kept < perm.counts).any()   # some assignments do drop

    sample = np.sort(np.random.default_rng(99).choice(T, size=SAMPLE, replace=False))
    forced = r.idx[sample].copy()
    forced[mism[sample]] = gi[sample][mism[sample]]
    keep = (perm.scatter_slot.reshape(T, k)[sample] >= 0).astype(np.float64)
    xs = f64(inp["x"][torch.from_numpy(sample)])
    rs = ref.route(oc, xs, ow.w_router, ow.b_router, ow.score_bias, forced)
    ps = ref.permute(rs.idx, E)
    y = ref.expert_outputs(oc, ref.prepare_routed_input(oc, xs, ow.w_down_latent), ps, ow.expert)
    z = ref.combine(y, ps.scatter_pos, rs.weights * keep)
    want = ref.restore_routed_output(oc, z, ow.w_up_latent, ow.rms_weight)
    assert_close_layer(out[sample], want, "olmoe capacity 1.0 sampled layer output")
