"""Full-size parity on the four large workloads, in the launch configuration
bench.py times (one moe_layer_forward with the library's own workspace plan).

All tokens: top-k indices against the float64 router (near-tie rule) and the
permutation, counts and offsets bit-exact against the oracle's counting sort
of the GPU's indices.  Sampled tokens: the layer output against the float64
oracle run on those tokens alone (tokens are independent), with the GPU's
choice adopted for near-tie tokens.  The sample is 96 random tokens plus,
for each of the 16 least-loaded experts that received any token, its first
and last 8 tokens: those experts' rows sit in mostly empty tail tiles of
the grouped GEMMs, which a random sample of a skewed load rarely reaches.
"""
import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from tests.oracle_bridge import assert_close_layer, check_topk, f64, oracle_config, oracle_weights
from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WORKLOADS, generate

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLE = 96
COLD_EXPERTS = 16
COLD_TOKENS = 8     # first and last this many tokens of each cold expert


def cold_expert_tokens(idx: np.ndarray, counts: np.ndarray) -> np.ndarray:
    """Tokens routed to the least-loaded experts that received any token (first and last few each)."""
    touched = np.nonzero(counts > 0)[0]
    cold = touched[np.argsort(counts[touched], kind="stable")[:COLD_EXPERTS]]
    toks = []
    for e in cold:
        t = np.nonzero((idx == e).any(axis=1))[0]
        toks.append(t[:COLD_TOKENS])
        toks.append(t[-COLD_TOKENS:])
    return np.unique(np.concatenate(toks)) if toks else np.zeros(0, np.int64)


@pytest.mark.parametrize("name", ["olmoe", "sigmoid_wide", "latent_prefill", "latent_decode"])
def test_full_size_workload(name):
    spec = WORKLOADS[name]
    T, E, k = spec.T, spec.num_experts, spec.top_k
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    x = inp["x"].cuda()
    ws = native.workspace(cfg, T)
    out = native.moe_layer_forward(cfg, wts, x, ws)
    assert native.moe_get_status() == 0
    inter = native.layer_intermediates(cfg, T, ws)
    gi = inter["idx"].cpu().numpy().astype(np.int64)
    counts = inter["counts"].cpu().numpy()
    offsets = inter["offsets"].cpu().numpy()
    gather = inter["gather_idx"].cpu().numpy()
    scatter = inter["scatter_idx"].cpu().numpy()
    out_np = out.double().cpu().numpy()
    del x

    oc, ow = oracle_config(spec), oracle_weights(spec, inp)
    r = ref.route(oc, f64(inp["x"]), ow.w_router, ow.b_router, ow.score_bias)
    mism = check_topk(gi, r.keys, r.idx, k)

    p = ref.permute(gi, E)
    np.testing.assert_array_equal(counts, p.counts)
    np.testing.assert_array_equal(offsets, p.offsets)
    np.testing.assert_array_equal(gather, p.gather_token)
    np.testing.assert_array_equal(scatter, p.scatter_pos)

    sample = np.random.default_rng(1234).choice(T, size=min(SAMPLE, T), replace=False)
    sample = np.union1d(sample, cold_expert_tokens(gi, counts))
    forced = r.idx[sample].copy()
    forced[mism[sample]] = gi[sample][mism[sample]]
    res = ref.layer_forward(oc, f64(inp["x"][torch.from_numpy(sample)]), ow, forced_idx=forced)
    assert_close_layer(out_np[sample], res.out, f"{name} sampled layer output")
