"""GPU parity of the MXFP8 experts (page "Как устроен Olmo-core 3: обучение больших MoE-моделей",
§"Rowwise FP8 и MXFP8", read as the OCP microscaling format) against the float64 oracle's MXFP8
path: the quantiser's codes and block scales bit-exact; the grouped experts and the layer within
the bars below.

The bars.  x_routed (bf16, non-latent) and the weights (bf16) quantise bit-exactly on both sides,
so GEMM 1 differs from the oracle by accumulation order only.  H is rounded to bf16 on both sides
from values that differ by that order; where the two fall on either side of a bf16 midpoint (a few
elements per row) an element's e4m3 code, or, if it is its block's amax on a power-of-two
boundary, its block's scale, may move by one step.  That perturbs 32 values at most, each by one
e4m3 step (2^-3 relative), so a token's output moves by far less than the rowwise-FP8 bar: the
tests ask for rel-L2 1e-2 over all outputs and at most half an e4m3 step (2^-4) per token."""
import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from tests.oracle_bridge import REL_L2, check_topk, f64, oracle_config, oracle_weights
from tests.test_gpu_parity import DESIGNED_COUNTS, designed_routing
from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WorkloadSpec, generate

pytestmark = pytest.mark.gpu

MX_TOKEN_REL = 2.0 ** -4


def assert_close_mx(got, want, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    tot = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert tot <= REL_L2, f"{what}: rel_l2={tot:.3e}"
    norms = np.linalg.norm(want, axis=1)
    live = norms > 0
    rels = np.linalg.norm(got - want, axis=1)[live] / norms[live]
    if rels.size:
        assert rels.max() <= MX_TOKEN_REL, f"{what}: row {int(np.nonzero(live)[0][rels.argmax()])} rel_l2={rels.max():.3e}"
    assert np.all(got[~live] == 0), f"{what}: rows with a zero oracle output are not zero"


@pytest.mark.parametrize("rows,cols,scale", [(1000, 256, 1.0), (77, 2048, 30.0), (5, 64, 1e-3), (9, 96, 1e-39)])
def test_mx_quantizer_bit_exact(rows, cols, scale):
    g = np.random.default_rng(rows + cols)
    x = torch.from_numpy((g.standard_normal((rows, cols)) * scale).astype(np.float32)).to(torch.bfloat16)
    x[min(3, rows - 1)] = 0.0                       # all-zero blocks: scale byte 0
    x[0, :32] = torch.tensor([448.0 * 2.0 ** -3] * 31 + [-1.0], dtype=torch.bfloat16)   # exact codes
    codes, scales = native.moe_quantize_mxfp8(x.cuda())
    assert native.moe_get_status() == 0
    want_q, want_e = ref.quantize_mx_e4m3(f64(x))
    assert scales.shape == (rows, native.mx_scale_ld(cols))
    np.testing.assert_array_equal(scales[:, :cols // 32].cpu().numpy().astype(np.int64), want_e)
    got_q = codes.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(got_q, want_q)


CASES = {
    "olmoe_like_small": WorkloadSpec("olmoe_like_small_mx", T=600, d_model=512, num_experts=8, top_k=2,
                                     hidden_size=256, gating="topk_softmax", expert_fp8=native.EXPERT_MXFP8, seed=81),
    "wide_ragged": WorkloadSpec("wide_ragged_mx", T=1500, d_model=640, num_experts=4, top_k=2, hidden_size=384,
                                gating="sigmoid", normalize_expert_weights=1.0, expert_fp8=native.EXPERT_MXFP8,
                                seed=82),
    "latent": WorkloadSpec("latent_mx", T=400, d_model=768, num_experts=16, top_k=4, hidden_size=256,
                           latent_dim=256, gating="sigmoid", skew=True, expert_fp8=native.EXPERT_MXFP8, seed=83),
    "capacity": WorkloadSpec("capacity_mx", T=512, d_model=256, num_experts=8, top_k=2, hidden_size=128,
                             gating="softmax", skew=True, capacity_factor=1.0, expert_fp8=native.EXPERT_MXFP8,
                             seed=84),
    # degenerate shapes: one token; one expert taking every row (several full tiles and a tail)
    "one_token": WorkloadSpec("one_token_mx", T=1, d_model=256, num_experts=4, top_k=2, hidden_size=128,
                              gating="softmax", expert_fp8=native.EXPERT_MXFP8, seed=86),
    "single_expert": WorkloadSpec("single_expert_mx", T=700, d_model=384, num_experts=1, top_k=1, hidden_size=256,
                                  gating="softmax", expert_fp8=native.EXPERT_MXFP8, seed=87),
}


def _layer(spec):
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp).quantize_experts_mxfp8()
    ws = native.workspace(cfg, spec.T)
    out = native.moe_layer_forward(cfg, wts, inp["x"].cuda(), ws)
    assert native.moe_get_status() == 0
    return inp, cfg, ws, out


def _capacity_mxfp8(oc, spec, x, ow, forced):
    """The oracle's capacity-limited layer with the MXFP8 experts on the kept slots (a padding
    slot is a zero row, whose MXFP8 output is zero, as in the bf16 capacity path)."""
    assert not oc.is_latent
    r = ref.route(oc, x, ow.w_router, ow.b_router, ow.score_bias, forced)
    cap = ref.expert_capacity(oc, x.shape[0], spec.capacity_factor)
    cperm = ref.permute_with_capacity(r.idx, oc.num_experts, cap)
    kept = cperm.kept.astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(kept)])
    slots = np.concatenate([np.arange(e * cap, e * cap + kept[e]) for e in range(oc.num_experts)]).astype(np.int64)
    dense = ref.Permutation(kept, offsets, cperm.slot_token[slots], None)
    y = np.zeros((oc.num_experts * cap, x.shape[1]))
    y[slots] = ref.expert_outputs_mxfp8(oc, x, dense, ow.expert)
    z = ref.combine_capacity(y, cperm.scatter_slot, r.weights)
    return ref.restore_routed_output(oc, z, ow.w_up_latent, ow.rms_weight)


@pytest.mark.parametrize("name", list(CASES))
def test_mxfp8_layer_forward(name):
    spec = CASES[name]
    inp, cfg, ws, out = _layer(spec)
    inter = native.layer_intermediates(cfg, spec.T, ws)
    oc, ow = oracle_config(spec), oracle_weights(spec, inp)
    r = ref.route(oc, f64(inp["x"]), ow.w_router, ow.b_router, ow.score_bias)
    gi = inter["idx"].cpu().numpy().astype(np.int64)
    mism = check_topk(gi, r.keys, r.idx, spec.top_k)
    forced = r.idx.copy()
    forced[mism] = gi[mism]
    if spec.capacity_factor > 0:
        want = _capacity_mxfp8(oc, spec, f64(inp["x"]), ow, forced)
    else:
        want = ref.layer_forward_mxfp8(oc, f64(inp["x"]), ow, forced_idx=forced)
    got = out.double().cpu().numpy()
    assert_close_mx(got, want, f"mxfp8 layer output ({name})")
    # and the MXFP8 layer stays close to the bf16 one
    dense = ref.layer_forward(oc, f64(inp["x"]), ow, forced_idx=forced).out if not spec.capacity_factor else None
    if dense is not None:
        assert np.linalg.norm(got - dense) / np.linalg.norm(dense) < 0.1


def test_mxfp8_grouped_swiglu_designed_counts():
    # every kind of group: empty, tail only, whole tiles only, whole tiles + tail
    spec = WorkloadSpec("designed_counts_mx", T=sum(DESIGNED_COUNTS), d_model=256,
                        num_experts=len(DESIGNED_COUNTS), top_k=1, hidden_size=256, gating="softmax",
                        expert_fp8=native.EXPERT_MXFP8, seed=85)
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp).quantize_experts_mxfp8()
    ws = native.workspace(cfg, spec.T)
    counts, offsets, gather, scatter = native.moe_permute(cfg, designed_routing(DESIGNED_COUNTS, 7), ws)
    xr = torch.from_numpy(np.random.default_rng(8).standard_normal((spec.T, spec.d_model), dtype=np.float32)).to(
        torch.bfloat16)
    y = native.moe_grouped_swiglu(cfg, wts, xr.cuda(), gather, offsets, ws)
    assert native.moe_get_status() == 0
    perm = ref.Permutation(counts.cpu().numpy(), offsets.cpu().numpy(), gather.cpu().numpy(), scatter.cpu().numpy())
    want = ref.expert_outputs_mxfp8(oracle_config(spec), f64(xr), perm, oracle_weights(spec, inp).expert)
    assert_close_mx(y.double().cpu().numpy(), want, "mxfp8 grouped swiglu, designed counts")


def test_mxfp8_config_checks():
    # 128-value k-tiles: d_model and hidden_size must be multiples of 128; no kept pre-activations
    bad = native.make_config(d_model=192, num_experts=4, top_k=1, hidden_size=128, expert_fp8=native.EXPERT_MXFP8)
    with pytest.raises(native.MoEError):
        native.moe_workspace_size(bad, 16)
    spec = CASES["olmoe_like_small"]
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)   # no MXFP8 weights
    ws = native.workspace(cfg, spec.T)
    with pytest.raises(native.MoEError):
        native.moe_layer_forward(cfg, wts, inp["x"].cuda(), ws)
    wts.quantize_experts_mxfp8()
    with pytest.raises(native.MoEError):
        native.moe_layer_forward_preact(cfg, wts, inp["x"].cuda(), ws)
