"""GPU parity of the load-balancing counters against the float64 oracle
(page "Как устроен Olmo-core 3: обучение больших MoE-моделей", §"Счётчики и
bias-корректировка").  Counters and the corrected score_bias are bit-exact
(one fp32 rounding on both sides); the imbalance ratio is within 1 fp32 ulp.
"""
import math

import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WORKLOADS, generate

pytestmark = pytest.mark.gpu


def _close_f32(got, want):
    if math.isnan(want):
        return math.isnan(got)
    return abs(got - want) <= 2.0 ** -22 * abs(want)


@pytest.mark.parametrize("E", [1, 7, 64, 896, 1024])
def test_accumulate_imbalance_and_bias_update(E):
    g = np.random.default_rng(E)
    accum_np = np.zeros(E, np.int64)
    accum = torch.zeros(E, dtype=torch.int64, device="cuda")
    for step in range(3):
        counts_np = g.integers(0, 5000, size=E).astype(np.int32)
        native.moe_accumulate_counts(torch.from_numpy(counts_np).cuda(), accum)
        accum_np = ref.accumulate_counts(accum_np, counts_np)
        imb = native.moe_load_imbalance(torch.from_numpy(counts_np).cuda())
        assert _close_f32(imb.item(), ref.load_imbalance(counts_np))
    assert native.moe_get_status() == 0
    np.testing.assert_array_equal(accum.cpu().numpy(), accum_np)
    assert _close_f32(native.moe_load_imbalance(accum).item(), ref.load_imbalance(accum_np))
    # make some experts sit exactly on the mean
    if E >= 4:
        accum_np[:2] = 1000
        accum_np[2:4] = 3000
        accum_np[4:] = 2000
        accum.copy_(torch.from_numpy(accum_np))
    bias_np = (g.standard_normal(E) * 0.01).astype(np.float32)
    bias = torch.from_numpy(bias_np.copy()).cuda()
    gamma = np.float32(0.001)
    native.moe_score_bias_update(accum, float(gamma), bias)
    want, zeroed = ref.score_bias_update(bias_np.astype(np.float64), accum_np, float(gamma))
    np.testing.assert_array_equal(bias.cpu().numpy(), want.astype(np.float32))
    np.testing.assert_array_equal(accum.cpu().numpy(), zeroed)


def test_imbalance_without_tokens_is_nan():
    assert math.isnan(native.moe_load_imbalance(torch.zeros(16, dtype=torch.int32, device="cuda")).item())


def test_bias_correction_loop_on_router_output():
    """router -> permute -> accumulate over two batches -> bias update, as between training steps."""
    spec = WORKLOADS["sigmoid_wide"].with_(T=1024, d_model=512, num_experts=64, hidden_size=128)
    inp = generate(spec, experts=False)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights(w_router=inp["w_router"].cuda(), w_up_gate=torch.empty(1, dtype=torch.bfloat16, device="cuda"),
                               w_out=torch.empty(1, dtype=torch.bfloat16, device="cuda"), score_bias=inp["score_bias"].cuda())
    ws = native.workspace(cfg, spec.T)
    accum = torch.zeros(spec.num_experts, dtype=torch.int64, device="cuda")
    accum_np = np.zeros(spec.num_experts, np.int64)
    x = inp["x"].cuda()
    for half in (x[:512].contiguous(), x[512:].contiguous()):
        _, idx, _ = native.moe_router(cfg, wts, half, ws)
        counts, _, _, _ = native.moe_permute(cfg, idx, ws)
        native.moe_accumulate_counts(counts, accum)
        accum_np = ref.accumulate_counts(accum_np, ref.permute(idx.cpu().numpy(), spec.num_experts).counts)
    bias0 = wts.score_bias.cpu().numpy()
    gamma = float(np.float32(0.001))                # the value the kernel receives (a float argument)
    native.moe_score_bias_update(accum, gamma, wts.score_bias)
    assert native.moe_get_status() == 0
    want, _ = ref.score_bias_update(bias0.astype(np.float64), accum_np, gamma)
    np.testing.assert_array_equal(wts.score_bias.cpu().numpy(), want.astype(np.float32))
    assert accum.abs().sum().item() == 0
