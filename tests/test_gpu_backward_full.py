"""Full-size parity of the training path bench.py times with --backward, on the OlmoE-shaped
layer: the layer forward that keeps the pre-activations, the combine backward and the experts
backward from the kept pre-activations, in the same launch configuration.

The oracle checks sampled outputs it can compute one by one (the backward of a row needs only
that row's token, its dy and its expert's weights):
  * the kept [u | g] of sampled rows;
  * dy and dweights of sampled tokens;
  * d x_routed of sampled tokens (the sum of their rows' input gradients, from the GPU's dy);
  * the weight gradients of sampled experts (all of their rows).
"""
import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from tests.oracle_bridge import REL_L2, f64, oracle_weights
from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WORKLOADS, generate

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def close(got, want, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    scale = max(np.abs(want).max(), 1e-30)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    mx = np.abs(got - want).max() / scale
    assert rel <= REL_L2 and mx <= 3e-2, f"{what}: rel_l2={rel:.3e} max_abs/scale={mx:.3e}"


def test_olmoe_training_path_sampled():
    spec = WORKLOADS["olmoe"]
    T, L, E, h, k = spec.T, spec.routed_dim, spec.num_experts, spec.hidden_size, spec.top_k
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    ws = native.workspace(cfg, T)
    x = inp["x"].cuda()
    _, pre = native.moe_layer_forward_preact(cfg, wts, x, ws)
    inter = native.layer_intermediates(cfg, T, ws)
    y, w = inter["y"], inter["weights"]
    gather, scatter, offsets = inter["gather_idx"], inter["scatter_idx"], inter["offsets"]
    dz = torch.from_numpy(np.random.default_rng(77).standard_normal((T, L), dtype=np.float32)).to(
        torch.bfloat16).cuda()
    dy, dw = native.moe_combine_backward(cfg, dz, y, scatter, w, gather_idx=gather)
    bws = native.backward_workspace(cfg, T)
    dx, dwug, dwo = native.moe_grouped_swiglu_backward_preact(cfg, wts, x, gather, offsets, scatter, dy, pre, bws)
    assert native.moe_get_status() == 0

    ow = oracle_weights(spec, inp)
    cache = {}

    def expert(e):   # float64 copies, made once per expert
        if e not in cache:
            cache[e] = ow.expert(e)
        return cache[e]

    x_np = f64(inp["x"])
    gather_np, scatter_np = gather.cpu().numpy(), scatter.cpu().numpy()
    off = offsets.cpu().numpy()
    expert_of_row = np.repeat(np.arange(E), np.diff(off))
    rng = np.random.default_rng(99)

    # kept pre-activations of sampled rows
    rows = np.sort(rng.choice(T * k, size=256, replace=False))
    pre_np = pre[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    want = np.stack([np.concatenate([x_np[gather_np[p]] @ expert(expert_of_row[p])[0].T,
                                     x_np[gather_np[p]] @ expert(expert_of_row[p])[1].T]) for p in rows])
    close(pre_np, want, "kept pre-activations (sampled rows)")

    # combine backward and the experts' input gradient of sampled tokens
    toks = np.sort(rng.choice(T, size=64, replace=False))
    y_np = y.double().cpu().numpy()
    dy_np = dy.double().cpu().numpy()
    dz_np = dz.double().cpu().numpy()
    w_np = w.double().cpu().numpy()
    dx_np = dx[torch.from_numpy(toks).cuda()].double().cpu().numpy()
    want_dy, want_dw, want_dx = [], [], []
    for t in toks:
        d_tok = np.zeros(L)
        for j in range(k):
            p = scatter_np[t * k + j]
            want_dy.append(w_np[t, j] * dz_np[t])
            want_dw.append(dz_np[t] @ y_np[p])
            w_up, w_gate, w_out = expert(expert_of_row[p])
            d_rows, _, _, _, _ = ref.swiglu_mlp_backward(x_np[t][None], w_up, w_gate, w_out, dy_np[p][None])
            d_tok += d_rows[0]
        want_dx.append(d_tok)
    ps = scatter_np.reshape(T, k)[toks].reshape(-1)
    close(dy_np[ps], np.stack(want_dy), "dy (sampled tokens)")
    close(dw.double().cpu().numpy()[toks].reshape(-1), np.array(want_dw), "dweights (sampled tokens)")
    close(dx_np, np.stack(want_dx), "dx_routed (sampled tokens)")

    # weight gradients of sampled experts, over all of their rows
    for e in sorted(rng.choice(E, size=2, replace=False).tolist()):
        lo, hi = int(off[e]), int(off[e + 1])
        w_up, w_gate, w_out = expert(e)
        _, dwu, dwg, dwo_e, _ = ref.swiglu_mlp_backward(x_np[gather_np[lo:hi]], w_up, w_gate, w_out, dy_np[lo:hi])
        close(dwug[e].double().cpu().numpy(), np.concatenate([dwu, dwg]), f"dW_up_gate[{e}]")
        close(dwo[e].double().cpu().numpy(), dwo_e, f"dW_out[{e}]")
