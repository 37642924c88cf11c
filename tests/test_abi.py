"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and its host-only functions (parameter counts, config checks, workspace plan)
behave as the header states.  No device entry point is called here.
"""
import os
import re

import pytest

from token_routing_expert_gb300 import native
from token_routing_expert_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(native.LIB_PATH):
        from token_routing_expert_gb300 import build
        build.build()
    return native.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe.h but not exported"
    assert sorted(native.EXPORTS) == names


def test_library_has_no_cuda_runtime_dependency():
    # the runtime is linked statically: loading needs neither a toolkit nor a GPU
    import subprocess
    out = subprocess.run(["ldd", native.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcudart" not in out


def _golden_rows():
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", "param_counts.txt")):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_param_counts_match_closed_forms(lib, row):
    name, D, L, E, k, h, router, total, active, proj = row[0], *map(int, row[1:])
    cfg = native.make_config(D, E, k, h, latent_dim=L)
    assert native.moe_num_params(cfg) == total
    assert native.moe_num_active_params(cfg) == active
    assert native.moe_latent_proj_params(cfg) == proj
    if L:
        assert native.moe_latent_proj_params(cfg, with_norm_gain=True) == proj + L
    cfgb = native.make_config(D, E, k, h, latent_dim=L, router_bias=True)
    assert native.moe_num_params(cfgb) == total + E


def test_validate_config_codes(lib):
    ok = native.make_config(256, 8, 2, 128)
    assert native.moe_validate_config(ok) == 0
    bad = [
        native.make_config(256, 8, 9, 128),               # top_k > num_experts
        native.make_config(0, 8, 2, 128),                 # d_model < 1
        native.make_config(256, 8, 2, 128, gating=7),     # unknown gating
        native.make_config(256, 8, 2, 128, normalize_expert_weights=-1.0),
        native.make_config(256, 8, 2, 128, latent_dim=-64),
    ]
    for c in bad:
        assert native.moe_validate_config(c) == 1
    unsupported = [
        native.make_config(200, 8, 2, 128),               # d_model not a multiple of 64
        native.make_config(256, 8, 2, 100),               # hidden not a multiple of 64
        native.make_config(256, 8, 2, 128, latent_dim=96),
        native.make_config(256, 2000, 2, 128),            # more experts than the kernels hold
        native.make_config(256, 64, 33, 128),             # top_k > 32
    ]
    for c in unsupported:
        assert native.moe_validate_config(c) == 2
    c = native.make_config(256, 8, 2, 128)
    c.activation = 1
    assert native.moe_validate_config(c) == 2
    # e4m3 expert modes: 0 bf16, 1 rowwise, 2 MXFP8; MXFP8 contracts 128-value k-tiles
    assert native.moe_validate_config(native.make_config(256, 8, 2, 128, expert_fp8=native.EXPERT_MXFP8)) == 0
    assert native.moe_validate_config(native.make_config(256, 8, 2, 128, expert_fp8=3)) == 1
    assert native.moe_validate_config(native.make_config(256, 8, 2, 128, expert_fp8=-1)) == 1
    for c in (native.make_config(192, 8, 2, 128, expert_fp8=native.EXPERT_MXFP8),   # d_model % 128
              native.make_config(256, 8, 2, 192, expert_fp8=native.EXPERT_MXFP8),   # hidden % 128
              native.make_config(256, 8, 2, 128, latent_dim=192, expert_fp8=native.EXPERT_MXFP8)):
        assert native.moe_validate_config(c) == 2
    assert native.moe_validate_config(native.make_config(192, 8, 2, 192, expert_fp8=native.EXPERT_FP8_ROWWISE)) == 0


def test_mx_scale_rows():
    # E8M0 scale rows: cols / 32 bytes, padded to 16 (a row's scales for four 128-value k-tiles are
    # read as one 16-byte word)
    assert [native.mx_scale_ld(c) for c in (32, 128, 512, 640, 1024, 2048, 7168)] == [16, 16, 16, 32, 32, 64, 224]


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workspace_plan(lib, name):
    spec = WORKLOADS[name]
    cfg = native.config_from_spec(spec)
    size = native.moe_workspace_size(cfg, spec.T)
    R, Lr = spec.rows, spec.routed_dim
    # at least: SwiGLU activations H and expert outputs Y (bf16) plus the routing arrays
    assert size >= R * (Lr + spec.hidden_size) * 2 + R * 16
    assert size % 256 == 0
    assert native.moe_workspace_size(cfg, 2 * spec.T) > size
    lay = native.moe_workspace_layout(cfg, spec.T)
    present = [o for o in lay if o >= 0]
    assert all(o % 256 == 0 and o < size for o in present)
    assert (lay[7] >= 0) == bool(spec.latent_dim) and (lay[9] >= 0) == bool(spec.latent_dim)
    # MXFP8 experts: H and Y in bf16 plus the permuted code rows of x_routed and H's codes
    if spec.routed_dim % 128 == 0 and spec.hidden_size % 128 == 0:
        mx = native.moe_workspace_size(native.config_from_spec(spec.with_(expert_fp8=native.EXPERT_MXFP8)), spec.T)
        assert mx >= R * (Lr + spec.hidden_size) * 3


def test_host_errors_enqueue_nothing(lib):
    import ctypes
    cfg = native.make_config(256, 8, 2, 128)
    out = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(cfg), -1, ctypes.byref(out)) == 1
    assert lib.moe_workspace_size(None, 4, ctypes.byref(out)) == 1
    # a device entry point with a workspace that is too small fails on the host
    w = native.moe_weights_t()
    assert lib.moe_router(ctypes.byref(cfg), ctypes.byref(w), 16, 4, None, 16, 16, 256, 8, None) == 3
    # misaligned workspace
    assert lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), 16, 4, 32, 1000, 1 << 30, None) == 3
    # empty batch: nothing to do, and no device needed
    assert lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), 16, 0, 32, None, 0, None) == 0
    assert native.load().moe_status_string(5) == b"device wait timed out"
    # MXFP8 quantiser: shape errors are found on the host; no rows is a no-op
    q = lib.moe_quantize_mxfp8
    assert q(16, 4, 48, 32, 32, 16, None) == 1        # cols not a multiple of 32
    assert q(16, 4, 64, 32, 32, 1, None) == 1         # scale_ld < cols / 32
    assert q(16, -1, 64, 32, 32, 16, None) == 1       # negative rows
    assert q(None, 4, 64, 32, 32, 16, None) == 1      # no input
    assert q(None, 0, 64, None, None, 16, None) == 0  # empty


def test_capacity_and_permuted_rows(lib):
    # roundup8(capacity_factor * top_k * T / E), hand-evaluated
    assert native.moe_expert_capacity(native.make_config(256, 64, 8, 128, capacity_factor=1.25), 8192) == 1280
    assert native.moe_expert_capacity(native.make_config(256, 8, 2, 128, capacity_factor=1.0), 100) == 32
    assert native.moe_expert_capacity(native.make_config(256, 8, 2, 128, capacity_factor=0.5), 100) == 16
    assert native.moe_expert_capacity(native.make_config(256, 8, 2, 128, capacity_factor=1.0), 96) == 24
    assert native.moe_expert_capacity(native.make_config(256, 8, 2, 128), 96) == 0        # dropless
    assert native.moe_permuted_rows(native.make_config(256, 8, 2, 128), 96) == 192
    assert native.moe_permuted_rows(native.make_config(256, 8, 2, 128, capacity_factor=1.0), 100) == 8 * 32
    assert native.moe_validate_config(native.make_config(256, 8, 2, 128, capacity_factor=-1.0)) == 1


def test_fp32_expert_rows_follow_the_weight_sum(lib):
    """moe_layer_expert_rows_fp32: fp32 y exactly when a non-latent bf16 layer's routing weights can
    add up to more than one per token."""
    f = native.moe_layer_expert_rows_fp32
    assert f(native.config_from_spec(WORKLOADS["sigmoid_wide"]))          # L1 then x 8
    assert not f(native.config_from_spec(WORKLOADS["olmoe"]))             # topk_softmax: sums to 1
    assert not f(native.config_from_spec(WORKLOADS["tiny"]))              # softmax, L1
    assert not f(native.config_from_spec(WORKLOADS["latent_prefill"]))    # latent: z is normalised
    assert not f(native.config_from_spec(WORKLOADS["sigmoid_wide"].with_(expert_fp8=1)))
    assert f(native.make_config(64, 16, 4, 64, gating="sigmoid"))        # sigmoid scores add up to 4
    assert f(native.make_config(64, 16, 4, 64, gating="softmax", normalize_expert_weights=2.0))   # up to 2
    assert not f(native.make_config(64, 16, 4, 64, gating="softmax", normalize_expert_weights=1.0))
    assert f(native.make_config(64, 16, 4, 64, gating="softmax", expert_weight_scale=1.5))
    assert not f(native.make_config(64, 16, 4, 64, gating="softmax", expert_weight_scale=0.5))
    assert f(native.make_config(64, 16, 4, 64, gating="topk_softmax", original_top_k=8))
    assert not f(native.make_config(64, 16, 1, 64, gating="sigmoid"))    # one sigmoid score: at most 1 + eps
