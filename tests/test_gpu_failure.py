"""Device-side failure path, without faulting the GPU: a bounded pipeline wait that nothing
completes gives up after its limit, reports MOE_ERR_TIMEOUT through the status word, and the
context stays usable (a layer forward right after still matches the oracle).  Host-side failures
(bad arguments, short workspaces, out-of-range indices) are covered in test_abi.py and
test_gpu_parity.py."""
import numpy as np
import pytest
from oracle import moe_ref as ref
from tests.oracle_bridge import assert_close_layer, f64, oracle_config, oracle_weights
from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WorkloadSpec, generate

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert native.moe_get_status(clear=True) == 0
    waited = native.moe_check_wait_timeout(50)
    assert 50 <= waited < 2000, waited
    assert native.moe_get_status() == 0          # the check cleared the status word again

    spec = WorkloadSpec("after_timeout", T=200, d_model=256, num_experts=8, top_k=2, hidden_size=128, seed=121)
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    ws = native.workspace(cfg, spec.T)
    out = native.moe_layer_forward(cfg, wts, inp["x"].cuda(), ws)
    assert native.moe_get_status() == 0
    idx = native.layer_intermediates(cfg, spec.T, ws)["idx"].cpu().numpy().astype(np.int64)
    want = ref.layer_forward(oracle_config(spec), f64(inp["x"]), oracle_weights(spec, inp), forced_idx=idx).out
    assert_close_layer(out.double().cpu().numpy(), want, "layer after the timeout check")


def test_wait_timeout_limits_are_checked_on_the_host():
    with pytest.raises(Exception):
        native.moe_check_wait_timeout(0)
    with pytest.raises(Exception):
        native.moe_check_wait_timeout(5000)
