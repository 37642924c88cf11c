"""moe_layer_forward_host_batches: batches in host memory, copies overlapped with the compute.
Every batch's output must equal moe_layer_forward's on the same input bit for bit (same kernels,
deterministic), whatever the overlap; the library's own convenience, with no counterpart on the page."""
import numpy as np
import pytest
import torch

from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WorkloadSpec, generate

pytestmark = pytest.mark.gpu

SPECS = [
    WorkloadSpec("host_small", T=300, d_model=256, num_experts=8, top_k=2, hidden_size=128, gating="softmax",
                 normalize_expert_weights=1.0, seed=41),
    WorkloadSpec("host_pair_latent", T=2000, d_model=768, num_experts=4, top_k=2, hidden_size=192, latent_dim=256,
                 gating="sigmoid", seed=42),
    WorkloadSpec("host_capacity", T=700, d_model=256, num_experts=8, top_k=2, hidden_size=128, gating="sigmoid",
                 skew=True, capacity_factor=1.0, seed=43),
    WorkloadSpec("host_fp8", T=900, d_model=512, num_experts=4, top_k=2, hidden_size=256, gating="topk_softmax",
                 expert_fp8=True, seed=44),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
@pytest.mark.parametrize("n_batches", [1, 2, 5])
def test_host_batches_match_device_forward(spec, n_batches):
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    if spec.expert_fp8:
        wts.quantize_experts_fp8()
    g = np.random.default_rng(spec.seed + n_batches)
    xs = [torch.from_numpy(g.standard_normal((spec.T, spec.d_model), dtype=np.float32)).to(torch.bfloat16).pin_memory()
          for _ in range(n_batches)]
    outs = [torch.full((spec.T, spec.d_model), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in xs]
    hws = native.host_workspace(cfg, spec.T)
    native.moe_layer_forward_host_batches(cfg, wts, xs, outs, hws)
    torch.cuda.current_stream().synchronize()
    assert native.moe_get_status() == 0
    ws = native.workspace(cfg, spec.T)
    for x, o in zip(xs, outs):
        want = native.moe_layer_forward(cfg, wts, x.cuda(), ws).cpu()
        assert torch.equal(o, want)


def test_host_batches_rejects_small_workspace():
    spec = SPECS[0]
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    x = [inp["x"].pin_memory()]
    out = [torch.empty_like(x[0]).pin_memory()]
    with pytest.raises(native.MoEError) as e:
        native.moe_layer_forward_host_batches(cfg, wts, x, out, native.workspace(cfg, spec.T))
    assert e.value.code == 3   # MOE_ERR_WORKSPACE: the staging buffers are missing
