"""GPU parity of the backward of the combine and of the grouped SwiGLU experts against the
float64 oracle (whose gradients are pinned by finite differences).  Inputs are the GPU's
own routing and permutation; gradients pass the layer bar (relative L2 <= 1e-2, max abs
<= 3e-2 after scaling by the tensor's largest magnitude), weight gradients of experts
without rows are exactly zero."""
import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from tests.oracle_bridge import REL_L2, f64, oracle_config, oracle_weights
from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WorkloadSpec, generate

pytestmark = pytest.mark.gpu

CASES = {
    "small": WorkloadSpec("small", T=300, d_model=256, num_experts=8, top_k=2, hidden_size=128, gating="softmax",
                          normalize_expert_weights=1.0, seed=51),
    "ragged_h_empty_experts": WorkloadSpec("ragged_h_empty_experts", T=200, d_model=512, num_experts=40, top_k=2,
                                           hidden_size=320, gating="sigmoid", skew=True, seed=52),
    "pair_tiles": WorkloadSpec("pair_tiles", T=2000, d_model=512, num_experts=4, top_k=2, hidden_size=256,
                               gating="topk_softmax", seed=53),
    "capacity": WorkloadSpec("capacity", T=400, d_model=256, num_experts=8, top_k=2, hidden_size=128,
                             gating="sigmoid", capacity_factor=0.75, seed=54),
    # the routed dimension is the latent one: the experts backward runs in it
    "latent_pair_tiles": WorkloadSpec("latent_pair_tiles", T=1600, d_model=384, num_experts=4, top_k=2,
                                      hidden_size=192, latent_dim=256, gating="sigmoid", skew=True, seed=55),
}


def close(got, want, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    scale = max(np.abs(want).max(), 1e-30)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    mx = np.abs(got - want).max() / scale
    assert rel <= REL_L2 and mx <= 3e-2, f"{what}: rel_l2={rel:.3e} max_abs/scale={mx:.3e}"


def check_preact(pre, x_np, gather_np, offsets, ow, E, h, what="preact"):
    """The kept pre-activations [u | g] against the oracle's projections of each row's token
    (zero rows for padding slots)."""
    pre = pre.double().cpu().numpy()
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        w_up, w_gate, _ = ow.expert(e)
        slots = gather_np[lo:hi]
        live = slots >= 0
        assert (pre[lo:hi][~live] == 0).all(), f"{what}: padding slots of expert {e} are not zero"
        if live.any():
            rows = x_np[slots[live]]
            close(pre[lo:hi][live], np.concatenate([rows @ w_up.T, rows @ w_gate.T], axis=1), f"{what}[{e}]")


@pytest.mark.parametrize("preact", [False, True], ids=["recompute", "saved_preact"])
@pytest.mark.parametrize("name", list(CASES))
def test_combine_and_experts_backward(name, preact):
    spec = CASES[name]
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    T, Lr, E, h = spec.T, spec.routed_dim, spec.num_experts, spec.hidden_size
    ws = native.workspace(cfg, T)
    x = inp["x"].cuda()
    _, idx, w = native.moe_router(cfg, wts, x, ws)
    counts, offsets, gather, scatter = native.moe_permute(cfg, idx, ws)
    x_in = x
    if spec.latent_dim:   # the experts' input is the latent projection of x
        x = native.moe_latent_down(cfg, wts, x_in, ws).clone()
    y = native.moe_grouped_swiglu(cfg, wts, x, gather, offsets, ws)
    pre = None
    if preact:
        y2, pre = native.moe_grouped_swiglu_preact(cfg, wts, x, gather, offsets, ws)
        assert torch.equal(y2, y), "keeping the pre-activations changed the forward"
    g = np.random.default_rng(spec.seed + 1)
    dz = torch.from_numpy(g.standard_normal((T, Lr), dtype=np.float32)).to(torch.bfloat16).cuda()
    dy, dw = native.moe_combine_backward(cfg, dz, y, scatter, w, gather_idx=gather)
    bws = native.backward_workspace(cfg, T)
    # the workspace starts dirty: nothing may depend on rows the backward does not write
    bws.fill_(0xFF)
    if preact:
        dx, dwug, dwo = native.moe_grouped_swiglu_backward_preact(cfg, wts, x, gather, offsets, scatter, dy, pre,
                                                                  bws)
    else:
        dx, dwug, dwo = native.moe_grouped_swiglu_backward(cfg, wts, x, gather, offsets, scatter, dy, bws)
    assert native.moe_get_status() == 0

    oc, ow = oracle_config(spec), oracle_weights(spec, inp)
    scatter_np, gather_np = scatter.cpu().numpy(), gather.cpu().numpy()
    y_np, w_np = y.double().cpu().numpy(), w.double().cpu().numpy()
    want_dy, want_dw = ref.combine_backward(f64(dz.cpu()), y_np, scatter_np, w_np)
    if spec.capacity_factor:
        assert (want_dy[gather_np < 0] == 0).all()
    close(dy.double().cpu().numpy(), want_dy, "dy")
    close(dw.double().cpu().numpy(), want_dw, "dweights")

    # experts' backward on the GPU's dy, in the dense (or slot) layout of the permutation
    dy_np = dy.double().cpu().numpy()
    x_np = x.double().cpu().numpy()
    if preact:
        check_preact(pre, x_np, gather_np, offsets.cpu().numpy(), ow, E, h)
    dx_want = np.zeros((T, Lr))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        rows = [p for p in range(lo, hi) if gather_np[p] >= 0]
        w_up, w_gate, w_out = ow.expert(e)
        got_wug = dwug[e].double().cpu().numpy()
        got_wo = dwo[e].double().cpu().numpy()
        if not rows:
            assert (got_wug == 0).all() and (got_wo == 0).all()
            continue
        tokens = gather_np[rows]
        d_rows, dwu, dwg, dwo_e, _ = ref.swiglu_mlp_backward(x_np[tokens], w_up, w_gate, w_out, dy_np[rows])
        np.add.at(dx_want, tokens, d_rows)
        close(got_wug, np.concatenate([dwu, dwg]), f"dW_up_gate[{e}]")
        close(got_wo, dwo_e, f"dW_out[{e}]")
    close(dx.double().cpu().numpy(), dx_want, "dx_routed")


ROUTER_CASES = {
    "softmax_p1": WorkloadSpec("softmax_p1", T=300, d_model=256, num_experts=8, top_k=2, hidden_size=128,
                               gating="softmax", normalize_expert_weights=1.0, seed=61),
    "topk_softmax_skew": WorkloadSpec("topk_softmax_skew", T=700, d_model=512, num_experts=40, top_k=6,
                                      hidden_size=128, gating="topk_softmax", skew=True, seed=62),
    "sigmoid_restore_bias": WorkloadSpec("sigmoid_restore_bias", T=500, d_model=512, num_experts=64, top_k=8,
                                         hidden_size=128, gating="sigmoid", sigmoid_stability_epsilon=1e-6,
                                         score_bias_std=0.01, normalize_expert_weights=1.0,
                                         restore_weight_scale=True, seed=63),
    "sigmoid_896_decode": WorkloadSpec("sigmoid_896_decode", T=64, d_model=1024, num_experts=896, top_k=8,
                                       hidden_size=128, gating="sigmoid", skew=True, original_top_k=16, seed=64),
    "few_experts": WorkloadSpec("few_experts", T=130, d_model=128, num_experts=6, top_k=6, hidden_size=64,
                                gating="softmax", expert_weight_scale=2.5, normalize_expert_weights=2.0, seed=65),
}


@pytest.mark.parametrize("name", list(ROUTER_CASES))
def test_router_backward(name):
    spec = ROUTER_CASES[name]
    inp = generate(spec, experts=False)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights(w_router=inp["w_router"].cuda(), w_up_gate=torch.empty(1, dtype=torch.bfloat16, device="cuda"),
                               w_out=torch.empty(1, dtype=torch.bfloat16, device="cuda"),
                               b_router=None if inp["b_router"] is None else inp["b_router"].cuda(),
                               score_bias=None if inp["score_bias"] is None else inp["score_bias"].cuda())
    T, D, E, k = spec.T, spec.d_model, spec.num_experts, spec.top_k
    x = inp["x"].cuda()
    ws = native.workspace(cfg, T)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    _, idx, _ = native.moe_router(cfg, wts, x, ws, logits=logits)
    g = np.random.default_rng(spec.seed + 5)
    dweights = torch.from_numpy(g.standard_normal((T, k), dtype=np.float32)).cuda()
    bws = native.backward_workspace(cfg, T)
    dl, dx, dw, db = native.moe_router_backward(cfg, wts, x, logits, idx, dweights, bws)
    assert native.moe_get_status() == 0
    oc, ow = oracle_config(spec), oracle_weights(spec, {**inp, "w_up_gate": None, "w_out": None})
    want_dl, want_dx, want_dw, want_db = ref.router_backward(oc, f64(inp["x"]), ow.w_router, ow.b_router,
                                                             ow.score_bias, idx.cpu().numpy(),
                                                             dweights.double().cpu().numpy())
    got_dl = dl.double().cpu().numpy()
    # fp32 recomputation of the same formulas
    assert np.abs(got_dl - want_dl).max() <= 1e-5 * np.abs(want_dl).max() + 1e-6
    close(dx.double().cpu().numpy(), want_dx, "router dx")
    close(dw.double().cpu().numpy(), want_dw, "dW_router")
    if spec.skew:
        close(db.double().cpu().numpy(), want_db, "db_router")


def test_layer_forward_preact_matches_forward():
    """The training forward returns the plain forward's output bit for bit and the pre-activations
    of the permutation it made (read back from the workspace)."""
    spec = CASES["pair_tiles"]
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    ws = native.workspace(cfg, spec.T)
    x = inp["x"].cuda()
    out = native.moe_layer_forward(cfg, wts, x, ws).clone()
    out2, pre = native.moe_layer_forward_preact(cfg, wts, x, ws)
    assert native.moe_get_status() == 0
    assert torch.equal(out, out2)
    inter = native.layer_intermediates(cfg, spec.T, ws)
    ow = oracle_weights(spec, inp)
    check_preact(pre, f64(inp["x"]), inter["gather_idx"].cpu().numpy(), inter["offsets"].cpu().numpy(), ow,
                 spec.num_experts, spec.hidden_size, "layer preact")


LATENT_CASES = {
    # (spec, with an RMSNorm gain)
    "norm_gain_small": (WorkloadSpec("norm_gain_small", T=300, d_model=384, num_experts=4, top_k=2, hidden_size=64,
                                     latent_dim=192, gating="softmax", seed=81), True),
    "norm_pair_tiles": (WorkloadSpec("norm_pair_tiles", T=1200, d_model=512, num_experts=4, top_k=2, hidden_size=64,
                                     latent_dim=256, gating="softmax", seed=82), False),
    "no_norm": (WorkloadSpec("no_norm", T=257, d_model=256, num_experts=4, top_k=2, hidden_size=64, latent_dim=128,
                             up_proj_norm=False, gating="softmax", seed=83), False),
}


@pytest.mark.parametrize("name", list(LATENT_CASES))
def test_latent_projection_backward(name):
    """Backward of the latent restore (RMSNorm + up-projection) and of the down-projection against
    the oracle's derivative of the forward definition, on random z, dout and dx_routed."""
    spec, with_gain = LATENT_CASES[name]
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    T, D, L = spec.T, spec.d_model, spec.latent_dim
    g = np.random.default_rng(spec.seed + 7)
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)   # noqa: E731
    gain = bf(1.0 + 0.3 * g.standard_normal(L)) if with_gain else None
    if gain is not None:
        wts.rms_weight = gain.cuda()
    z, dout, dxr = bf(g.standard_normal((T, L))), bf(g.standard_normal((T, D))), bf(g.standard_normal((T, L)))
    bws = native.backward_workspace(cfg, T)
    bws.fill_(0xFF)
    dz, dw_up, dg = native.moe_latent_restore_backward(cfg, wts, z.cuda(), dout.cuda(), bws)
    dx, dw_down = native.moe_latent_down_backward(cfg, wts, inp["x"].cuda(), dxr.cuda(), bws)
    assert native.moe_get_status() == 0
    oc = oracle_config(spec)
    want_dz, want_dwu, want_dg = ref.restore_routed_output_backward(oc, f64(z), f64(inp["w_up_latent"]), f64(dout),
                                                                    None if gain is None else f64(gain))
    close(dz.double().cpu().numpy(), want_dz, "dz")
    close(dw_up.double().cpu().numpy(), want_dwu, "dW_up")
    if spec.up_proj_norm:
        close(dg.double().cpu().numpy(), want_dg, "dgamma")
    else:
        assert dg is None
    want_dx, want_dwd = ref.prepare_routed_input_backward(f64(inp["x"]), f64(inp["w_down"]), f64(dxr))
    close(dx.double().cpu().numpy(), want_dx, "dx (latent down-projection)")
    close(dw_down.double().cpu().numpy(), want_dwd, "dW_down")


LAYER_CASES = {
    # (spec, with an RMSNorm gain)
    "router_and_score_bias": (WorkloadSpec("router_and_score_bias", T=600, d_model=256, num_experts=8, top_k=2,
                                           hidden_size=128, gating="sigmoid", skew=True, score_bias_std=0.01,
                                           normalize_expert_weights=1.0, seed=91), False),
    "latent_gain": (WorkloadSpec("latent_gain", T=400, d_model=384, num_experts=6, top_k=2, hidden_size=64,
                                 latent_dim=192, gating="topk_softmax", seed=92), True),
    "latent_pair_tiles": (WorkloadSpec("latent_pair_tiles", T=1600, d_model=384, num_experts=4, top_k=2,
                                       hidden_size=128, latent_dim=256, gating="softmax", seed=93), False),
    # dropped assignments: their rows are padding slots, their weights get no gradient from the experts
    "capacity": (WorkloadSpec("capacity_layer", T=500, d_model=256, num_experts=8, top_k=2, hidden_size=128,
                              gating="sigmoid", skew=True, capacity_factor=0.75, seed=94), False),
    # degenerate shapes: one token (most experts empty), one expert, every expert chosen by every token
    "one_token": (WorkloadSpec("one_token_bwd", T=1, d_model=256, num_experts=8, top_k=2, hidden_size=128,
                               gating="softmax", normalize_expert_weights=1.0, seed=95), False),
    "single_expert": (WorkloadSpec("single_expert_bwd", T=130, d_model=128, num_experts=1, top_k=1,
                                   hidden_size=64, gating="sigmoid", seed=96), False),
    "all_experts": (WorkloadSpec("all_experts_bwd", T=150, d_model=192, num_experts=6, top_k=6, hidden_size=64,
                                 gating="topk_softmax", seed=97), False),
}


@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_layer_backward(name):
    """moe_layer_backward after moe_layer_forward_preact: every gradient against the oracle's chain of
    derivatives on the forward's own routing and expert outputs, and bit for bit against the
    library's steps called one by one."""
    spec, with_gain = LAYER_CASES[name]
    inp = generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    T, D, E, k = spec.T, spec.d_model, spec.num_experts, spec.top_k
    latent = bool(spec.latent_dim)
    g = np.random.default_rng(spec.seed + 3)
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)   # noqa: E731
    gain = bf(1.0 + 0.3 * g.standard_normal(spec.latent_dim)) if with_gain else None
    if gain is not None:
        wts.rms_weight = gain.cuda()
    x = inp["x"].cuda()
    ws = native.workspace(cfg, T)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    out, pre = native.moe_layer_forward_preact(cfg, wts, x, ws, logits=logits)
    dout = bf(g.standard_normal((T, D))).cuda()
    bws = native.layer_backward_workspace(cfg, T)
    bws.fill_(0xFF)
    dx, grads = native.moe_layer_backward(cfg, wts, x, ws, pre, logits, dout, bws)
    assert native.moe_get_status() == 0
    inter = native.layer_intermediates(cfg, T, ws)

    # the same steps called one by one
    sws = native.backward_workspace(cfg, T)
    y, w, sc, ga, off = inter["y"], inter["weights"], inter["scatter_idx"], inter["gather_idx"], inter["offsets"]
    dz = dout
    if latent:
        z = native.moe_combine(cfg, y, sc, w, T)
        dz, dwu, dg = native.moe_latent_restore_backward(cfg, wts, z, dout, sws)
        assert torch.equal(dwu, grads["dw_up_latent"]) and torch.equal(dg, grads["drms_weight"])
    dy, dwts = native.moe_combine_backward(cfg, dz, y, sc, w, gather_idx=ga)
    xr = inter["x_routed"] if latent else x
    dxr, dwug, dwo = native.moe_grouped_swiglu_backward_preact(cfg, wts, xr, ga, off, sc, dy, pre, sws)
    assert torch.equal(dwug, grads["dw_up_gate"]) and torch.equal(dwo, grads["dw_out"])
    dx_e = dxr
    if latent:
        dx_e, dwd = native.moe_latent_down_backward(cfg, wts, x, dxr, sws)
        assert torch.equal(dwd, grads["dw_down_latent"])
    _, dx_r, dwr, dbr = native.moe_router_backward(cfg, wts, x, logits, inter["idx"], dwts, sws)
    assert torch.equal(dwr, grads["dw_router"])
    if cfg.router_bias:
        assert torch.equal(dbr, grads["db_router"])
    assert torch.equal((dx_e.float() + dx_r.float()).to(torch.bfloat16), dx)

    # the oracle's chain of derivatives on the forward's routing and expert outputs
    oc, ow = oracle_config(spec), oracle_weights(spec, inp)
    gamma = None if gain is None else f64(gain)
    x_np, y_np, w_np = f64(inp["x"]), y.double().cpu().numpy(), w.double().cpu().numpy()
    sc_np, ga_np = sc.cpu().numpy(), ga.cpu().numpy()
    perm = ref.Permutation(inter["counts"].cpu().numpy(), off.cpu().numpy(), ga_np, sc_np)
    dz_np = f64(dout.cpu())
    if latent:
        z_np = ref.combine(y_np, sc_np, w_np)
        dz_np, want_dwu, want_dg = ref.restore_routed_output_backward(oc, z_np, ow.w_up_latent, dz_np, gamma)
        close(grads["dw_up_latent"].double().cpu().numpy(), want_dwu, "dW_up")
        close(grads["drms_weight"].double().cpu().numpy(), want_dg, "dgamma")
    want_dy, want_dwts = ref.combine_backward(dz_np, y_np, sc_np, w_np)
    xr_np = xr.double().cpu().numpy()
    if spec.capacity_factor:
        # capacity slots: padding slots (gather -1) are no rows; the oracle's experts backward is the
        # dropless one, so it runs on each expert's live slots
        want_dxr, want_grads = np.zeros_like(xr_np), {}
        for e in range(E):
            lo, hi = int(off[e]), int(off[e + 1])
            live = [q for q in range(lo, hi) if ga_np[q] >= 0]
            w_up, w_gate, w_out = ow.expert(e)
            if not live:
                want_grads[e] = (np.zeros_like(w_up), np.zeros_like(w_gate), np.zeros_like(w_out))
                continue
            d_rows, dwu, dwg, dwo_e, _ = ref.swiglu_mlp_backward(xr_np[ga_np[live]], w_up, w_gate, w_out,
                                                                  want_dy[live])
            np.add.at(want_dxr, ga_np[live], d_rows)
            want_grads[e] = (dwu, dwg, dwo_e)
    else:
        want_dxr, want_grads = ref.experts_backward(oc, xr_np, perm, ow.expert, want_dy)
    for e in range(E):
        close(grads["dw_up_gate"][e].double().cpu().numpy(), np.concatenate(want_grads[e][:2]), f"dW_up_gate[{e}]")
        close(grads["dw_out"][e].double().cpu().numpy(), want_grads[e][2], f"dW_out[{e}]")
    want_dx = want_dxr
    if latent:
        want_dx, want_dwd = ref.prepare_routed_input_backward(x_np, ow.w_down_latent, want_dxr)
        close(grads["dw_down_latent"].double().cpu().numpy(), want_dwd, "dW_down")
    _, want_dx_r, want_dwr, want_dbr = ref.router_backward(oc, x_np, ow.w_router, ow.b_router, ow.score_bias,
                                                           inter["idx"].cpu().numpy(), want_dwts)
    close(grads["dw_router"].double().cpu().numpy(), want_dwr, "dW_router")
    if cfg.router_bias:
        close(grads["db_router"].double().cpu().numpy(), want_dbr, "db_router")
    close(dx.double().cpu().numpy(), want_dx + want_dx_r, "dx (layer)")
