"""ctypes binding of ``libmoe_gb300.so``: argument marshalling only.

Every function here has the name of the C entry point it calls and takes
torch CUDA tensors; all arithmetic happens in the library's kernels.  There
is no fallback: if the library is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from .workloads import GATING_NAMES, WorkloadSpec

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_BOUNDS", 7: "MOE_ERR_NO_DEVICE"}


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({_status_string(code)})")


class moe_config_t(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("hidden_size", ctypes.c_int32), ("latent_dim", ctypes.c_int32), ("up_proj_norm", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("gating", ctypes.c_int32),
                ("sigmoid_stability_epsilon", ctypes.c_float), ("normalize_expert_weights", ctypes.c_float),
                ("restore_weight_scale", ctypes.c_int32), ("expert_weight_scale", ctypes.c_float),
                ("original_top_k", ctypes.c_int32), ("router_bias", ctypes.c_int32),
                ("has_score_bias", ctypes.c_int32), ("activation", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("expert_fp8", ctypes.c_int32)]


class moe_weights_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_router", "b_router", "score_bias", "w_down_latent",
                                                  "w_up_latent", "rms_weight", "w_up_gate", "w_out",
                                                  "w_up_gate_fp8", "w_up_gate_scale", "w_out_fp8", "w_out_scale",
                                                  "w_up_gate_mx_scale", "w_out_mx_scale")]


class moe_grads_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("dw_router", "db_router", "dw_up_gate", "dw_out", "dw_down_latent",
                                                  "dw_up_latent", "drms_weight")]


EXPORTS = ["moe_quantize_rowwise_fp8", "moe_expert_capacity", "moe_permuted_rows", "moe_validate_config", "moe_num_params", "moe_num_active_params", "moe_latent_proj_params",
           "moe_workspace_size", "moe_router", "moe_permute", "moe_grouped_swiglu", "moe_combine",
           "moe_latent_down", "moe_latent_restore", "moe_layer_forward", "moe_layer_forward_staged",
           "moe_layer_forward_launches", "moe_workspace_layout", "moe_get_status", "moe_status_string",
           "moe_permute_noalloc", "moe_accumulate_counts", "moe_load_imbalance", "moe_score_bias_update",
           "moe_backward_workspace_size", "moe_combine_backward", "moe_grouped_swiglu_backward",
           "moe_router_backward", "moe_host_workspace_size", "moe_layer_forward_host_batches",
           "moe_grouped_swiglu_preact", "moe_layer_forward_preact", "moe_grouped_swiglu_backward_preact",
           "moe_latent_restore_backward", "moe_latent_down_backward", "moe_layer_backward_workspace_size",
           "moe_layer_backward", "moe_check_wait_timeout", "moe_quantize_mxfp8", "moe_layer_expert_rows_fp32"]

_lib = None


def load() -> ctypes.CDLL:
    """Loads the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with token_routing_expert_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, SZ, VP = ctypes.POINTER, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
    cfgp, wp = P(moe_config_t), P(moe_weights_t)
    sig = {
        "moe_validate_config": [cfgp],
        "moe_num_params": [cfgp, P(I64)],
        "moe_num_active_params": [cfgp, P(I64)],
        "moe_latent_proj_params": [cfgp, ctypes.c_int, P(I64)],
        "moe_workspace_size": [cfgp, I64, P(SZ)],
        "moe_expert_capacity": [cfgp, I64, P(I64)],
        "moe_quantize_rowwise_fp8": [VP, I64, ctypes.c_int32, VP, VP, VP],
        "moe_permuted_rows": [cfgp, I64, P(I64)],
        "moe_router": [cfgp, wp, VP, I64, VP, VP, VP, VP, SZ, VP],
        "moe_permute": [cfgp, VP, I64, VP, VP, VP, VP, VP, SZ, VP],
        "moe_grouped_swiglu": [cfgp, wp, VP, VP, VP, I64, VP, VP, SZ, VP],
        "moe_grouped_swiglu_preact": [cfgp, wp, VP, VP, VP, I64, VP, VP, VP, SZ, VP],
        "moe_combine": [cfgp, VP, VP, VP, I64, VP, VP],
        "moe_latent_down": [cfgp, wp, VP, I64, VP, VP, SZ, VP],
        "moe_latent_restore": [cfgp, wp, VP, I64, VP, VP, SZ, VP],
        "moe_layer_forward": [cfgp, wp, VP, I64, VP, VP, SZ, VP],
        "moe_layer_forward_preact": [cfgp, wp, VP, I64, VP, VP, VP, VP, SZ, VP],
        "moe_layer_forward_staged": [cfgp, wp, VP, I64, VP, VP, SZ, VP, P(VP)],
        "moe_layer_forward_launches": [cfgp, I64, P(ctypes.c_int32)],
        "moe_host_workspace_size": [cfgp, I64, P(SZ)],
        "moe_layer_forward_host_batches": [cfgp, wp, P(VP), P(VP), ctypes.c_int32, I64, VP, SZ, VP],
        "moe_workspace_layout": [cfgp, I64, P(I64)],
        "moe_layer_expert_rows_fp32": [cfgp, P(ctypes.c_int32)],
        "moe_get_status": [VP, P(ctypes.c_int32), ctypes.c_int],
        "moe_status_string": [ctypes.c_int],
        "moe_permute_noalloc": [cfgp, VP, I64, VP, VP, VP, VP, VP],
        "moe_accumulate_counts": [VP, ctypes.c_int32, VP, VP],
        "moe_backward_workspace_size": [cfgp, I64, P(SZ)],
        "moe_router_backward": [cfgp, wp, VP, I64, VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP],
        "moe_latent_restore_backward": [cfgp, wp, VP, I64, VP, VP, VP, VP, VP, SZ, VP],
        "moe_latent_down_backward": [cfgp, wp, VP, I64, VP, VP, VP, VP, SZ, VP],
        "moe_layer_backward_workspace_size": [cfgp, I64, P(SZ)],
        "moe_check_wait_timeout": [ctypes.c_int32, P(ctypes.c_int32), VP],
        "moe_quantize_mxfp8": [VP, I64, ctypes.c_int32, VP, VP, ctypes.c_int32, VP],
        "moe_layer_backward": [cfgp, wp, VP, I64, VP, SZ, VP, VP, VP, VP, P(moe_grads_t), VP, SZ, VP],
        "moe_combine_backward": [cfgp, VP, VP, VP, VP, VP, I64, VP, VP, VP],
        "moe_grouped_swiglu_backward": [cfgp, wp, VP, VP, VP, VP, I64, VP, VP, VP, VP, VP, SZ, VP],
        "moe_grouped_swiglu_backward_preact": [cfgp, wp, VP, VP, VP, VP, I64, VP, VP, VP, VP, VP, VP, SZ, VP],
        "moe_load_imbalance": [VP, ctypes.c_int32, ctypes.c_int32, VP, VP],
        "moe_score_bias_update": [VP, ctypes.c_int32, ctypes.c_float, VP, VP],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "moe_status_string" else ctypes.c_int
    _lib = lib
    return lib


def _status_string(code: int) -> str:
    try:
        return load().moe_status_string(code).decode()
    except Exception:  # noqa: BLE001 - only for messages
        return "?"


def _check(code: int, where: str) -> None:
    if code != MOE_OK:
        raise MoEError(code, where)


# moe_config_t.expert_fp8: operands of the experts' GEMMs
EXPERT_BF16, EXPERT_FP8_ROWWISE, EXPERT_MXFP8 = 0, 1, 2


def make_config(d_model, num_experts, top_k, hidden_size, latent_dim=0, up_proj_norm=True, rms_eps=1e-6,
                gating="softmax", sigmoid_stability_epsilon=0.0, normalize_expert_weights=0.0,
                restore_weight_scale=False, expert_weight_scale=0.0, original_top_k=0, router_bias=False,
                has_score_bias=False, capacity_factor=0.0, expert_fp8=False) -> moe_config_t:
    g = GATING_NAMES[gating] if isinstance(gating, str) else int(gating)
    return moe_config_t(d_model, num_experts, top_k, hidden_size, latent_dim, int(up_proj_norm), rms_eps, g,
                        sigmoid_stability_epsilon, normalize_expert_weights, int(restore_weight_scale),
                        expert_weight_scale, original_top_k, int(router_bias), int(has_score_bias), 0,
                        capacity_factor, int(expert_fp8))


def config_from_spec(spec: WorkloadSpec) -> moe_config_t:
    return make_config(spec.d_model, spec.num_experts, spec.top_k, spec.hidden_size, spec.latent_dim,
                       spec.up_proj_norm, spec.rms_eps, spec.gating, spec.sigmoid_stability_epsilon,
                       spec.normalize_expert_weights, spec.restore_weight_scale, spec.expert_weight_scale,
                       spec.original_top_k, spec.skew, spec.score_bias_std > 0, spec.capacity_factor,
                       spec.expert_fp8)


# ---------------------------------------------------------------------------
# host-only functions
# ---------------------------------------------------------------------------

def moe_validate_config(cfg: moe_config_t) -> int:
    return load().moe_validate_config(ctypes.byref(cfg))


def moe_num_params(cfg: moe_config_t) -> int:
    out = ctypes.c_int64()
    _check(load().moe_num_params(ctypes.byref(cfg), ctypes.byref(out)), "moe_num_params")
    return out.value


def moe_num_active_params(cfg: moe_config_t) -> int:
    out = ctypes.c_int64()
    _check(load().moe_num_active_params(ctypes.byref(cfg), ctypes.byref(out)), "moe_num_active_params")
    return out.value


def moe_latent_proj_params(cfg: moe_config_t, with_norm_gain: bool = False) -> int:
    out = ctypes.c_int64()
    _check(load().moe_latent_proj_params(ctypes.byref(cfg), int(with_norm_gain), ctypes.byref(out)),
           "moe_latent_proj_params")
    return out.value


def moe_workspace_size(cfg: moe_config_t, T: int) -> int:
    out = ctypes.c_size_t()
    _check(load().moe_workspace_size(ctypes.byref(cfg), T, ctypes.byref(out)), "moe_workspace_size")
    return out.value


def moe_expert_capacity(cfg: moe_config_t, T: int) -> int:
    out = ctypes.c_int64()
    _check(load().moe_expert_capacity(ctypes.byref(cfg), T, ctypes.byref(out)), "moe_expert_capacity")
    return out.value


def moe_permuted_rows(cfg: moe_config_t, T: int) -> int:
    out = ctypes.c_int64()
    _check(load().moe_permuted_rows(ctypes.byref(cfg), T, ctypes.byref(out)), "moe_permuted_rows")
    return out.value


def moe_layer_expert_rows_fp32(cfg: moe_config_t) -> bool:
    out = ctypes.c_int32()
    _check(load().moe_layer_expert_rows_fp32(ctypes.byref(cfg), ctypes.byref(out)), "moe_layer_expert_rows_fp32")
    return bool(out.value)


def moe_workspace_layout(cfg: moe_config_t, T: int):
    arr = (ctypes.c_int64 * 10)()
    _check(load().moe_workspace_layout(ctypes.byref(cfg), T, arr), "moe_workspace_layout")
    return list(arr)


# ---------------------------------------------------------------------------
# device entry points
# ---------------------------------------------------------------------------

def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class DeviceWeights:
    """The layer's weights on the device (bf16, fp32 for biases), kept alive by this object."""

    w_router: torch.Tensor
    w_up_gate: torch.Tensor
    w_out: torch.Tensor
    b_router: Optional[torch.Tensor] = None
    score_bias: Optional[torch.Tensor] = None
    w_down_latent: Optional[torch.Tensor] = None
    w_up_latent: Optional[torch.Tensor] = None
    rms_weight: Optional[torch.Tensor] = None
    w_up_gate_fp8: Optional[torch.Tensor] = None
    w_up_gate_scale: Optional[torch.Tensor] = None
    w_out_fp8: Optional[torch.Tensor] = None
    w_out_scale: Optional[torch.Tensor] = None
    w_up_gate_mx_scale: Optional[torch.Tensor] = None
    w_out_mx_scale: Optional[torch.Tensor] = None

    def quantize_experts_fp8(self, stream=None) -> "DeviceWeights":
        """Pre-quantises the expert weights row by row to e4m3 (moe_quantize_rowwise_fp8)."""
        ug, wo = self.w_up_gate, self.w_out
        self.w_up_gate_fp8, self.w_up_gate_scale = moe_quantize_rowwise_fp8(ug.reshape(-1, ug.shape[-1]), stream=stream)
        self.w_out_fp8, self.w_out_scale = moe_quantize_rowwise_fp8(wo.reshape(-1, wo.shape[-1]), stream=stream)
        return self

    def quantize_experts_mxfp8(self, stream=None) -> "DeviceWeights":
        """Pre-quantises the expert weights to MXFP8 along their contraction (moe_quantize_mxfp8)."""
        ug, wo = self.w_up_gate, self.w_out
        self.w_up_gate_fp8, self.w_up_gate_mx_scale = moe_quantize_mxfp8(ug.reshape(-1, ug.shape[-1]), stream=stream)
        self.w_out_fp8, self.w_out_mx_scale = moe_quantize_mxfp8(wo.reshape(-1, wo.shape[-1]), stream=stream)
        return self

    @staticmethod
    def from_inputs(inp, device="cuda") -> "DeviceWeights":
        def dev(name):
            t = inp.get(name)
            return None if t is None else t.to(device).contiguous()

        return DeviceWeights(w_router=dev("w_router"), w_up_gate=dev("w_up_gate"), w_out=dev("w_out"),
                             b_router=dev("b_router"), score_bias=dev("score_bias"),
                             w_down_latent=dev("w_down"), w_up_latent=dev("w_up_latent"),
                             rms_weight=dev("rms_weight"))

    def struct(self) -> moe_weights_t:
        bf, f32 = torch.bfloat16, torch.float32
        return moe_weights_t(
            _ptr(self.w_router, bf, "w_router"), _ptr(self.b_router, f32, "b_router"),
            _ptr(self.score_bias, f32, "score_bias"), _ptr(self.w_down_latent, bf, "w_down_latent"),
            _ptr(self.w_up_latent, bf, "w_up_latent"), _ptr(self.rms_weight, bf, "rms_weight"),
            _ptr(self.w_up_gate, bf, "w_up_gate"), _ptr(self.w_out, bf, "w_out"),
            _ptr(self.w_up_gate_fp8, torch.uint8, "w_up_gate_fp8"), _ptr(self.w_up_gate_scale, f32, "w_up_gate_scale"),
            _ptr(self.w_out_fp8, torch.uint8, "w_out_fp8"), _ptr(self.w_out_scale, f32, "w_out_scale"),
            _ptr(self.w_up_gate_mx_scale, torch.uint8, "w_up_gate_mx_scale"),
            _ptr(self.w_out_mx_scale, torch.uint8, "w_out_mx_scale"))


def moe_quantize_rowwise_fp8(x, codes=None, scales=None, stream=None):
    """Rowwise e4m3 codes (uint8, same shape) and fp32 row scales of a 2-D bf16 CUDA tensor."""
    rows, cols = x.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=x.device) if codes is None else codes
    scales = torch.empty(rows, dtype=torch.float32, device=x.device) if scales is None else scales
    _check(load().moe_quantize_rowwise_fp8(_ptr(x, torch.bfloat16, "x"), rows, cols, _ptr(codes, torch.uint8, "codes"),
                                           _ptr(scales, torch.float32, "scales"), _stream(stream)),
           "moe_quantize_rowwise_fp8")
    return codes, scales


def workspace(cfg: moe_config_t, T: int, device="cuda") -> torch.Tensor:
    """A device workspace of moe_workspace_size bytes (torch allocations are 256-byte aligned)."""
    return torch.empty(max(1, moe_workspace_size(cfg, T)), dtype=torch.uint8, device=device)


def moe_router(cfg, weights: DeviceWeights, x, ws, logits=None, idx=None, w=None, stream=None):
    T = x.shape[0]
    dev = x.device
    idx = torch.empty((T, cfg.top_k), dtype=torch.int32, device=dev) if idx is None else idx
    w = torch.empty((T, cfg.top_k), dtype=torch.float32, device=dev) if w is None else w
    ws_ = weights.struct()
    _check(load().moe_router(ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x, torch.bfloat16, "x"), T,
                             _ptr(logits, torch.float32, "logits"), _ptr(idx, torch.int32, "idx"),
                             _ptr(w, torch.float32, "weights"), _ptr(ws, None, "ws"), ws.numel(), _stream(stream)),
           "moe_router")
    return logits, idx, w


def _check_permute_outputs(cfg, idx, counts, offsets, gather_idx, scatter_idx, rows, what):
    """The C ABI cannot see buffer sizes: undersized outputs would be written past their end."""
    T = idx.shape[0]
    if idx.dim() != 2 or idx.shape[1] != cfg.top_k:
        raise ValueError(f"{what}: idx must be (T, top_k={cfg.top_k}), got {tuple(idx.shape)}")
    E, R = cfg.num_experts, T * cfg.top_k
    for name, t, n in (("counts", counts, E), ("offsets", offsets, E + 1), ("gather_idx", gather_idx, rows),
                       ("scatter_idx", scatter_idx, R)):
        if t.numel() < n:
            raise ValueError(f"{what}: {name} holds {t.numel()} entries, needs {n}")
        if t.device != idx.device:
            raise ValueError(f"{what}: {name} is on {t.device}, idx on {idx.device}")
    if idx.is_cuda and idx.device.index != torch.cuda.current_device():
        raise ValueError(f"{what}: tensors are on {idx.device}, the current device is cuda:{torch.cuda.current_device()}")


def moe_permute(cfg, idx, ws, counts=None, offsets=None, gather_idx=None, scatter_idx=None, stream=None):
    T = idx.shape[0]
    R = T * cfg.top_k
    rows = moe_permuted_rows(cfg, T)
    dev = idx.device
    E = cfg.num_experts
    counts = torch.empty(E, dtype=torch.int32, device=dev) if counts is None else counts
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    gather_idx = torch.empty(max(rows, 1), dtype=torch.int32, device=dev) if gather_idx is None else gather_idx
    scatter_idx = torch.empty(max(R, 1), dtype=torch.int32, device=dev) if scatter_idx is None else scatter_idx
    _check_permute_outputs(cfg, idx, counts, offsets, gather_idx, scatter_idx, rows, "moe_permute")
    _check(load().moe_permute(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"), T,
                              _ptr(counts, torch.int32, "counts"), _ptr(offsets, torch.int32, "offsets"),
                              _ptr(gather_idx, torch.int32, "gather_idx"), _ptr(scatter_idx, torch.int32, "scatter_idx"),
                              _ptr(ws, None, "ws"), ws.numel(), _stream(stream)), "moe_permute")
    return counts, offsets, gather_idx[:rows], scatter_idx[:R]


def moe_permute_noalloc(cfg, idx, counts, offsets, gather_idx, scatter_idx, stream=None):
    """moe_permute with no workspace (the library's static scratch); outputs are the caller's tensors."""
    T = idx.shape[0]
    _check_permute_outputs(cfg, idx, counts, offsets, gather_idx, scatter_idx, T * cfg.top_k, "moe_permute_noalloc")
    _check(load().moe_permute_noalloc(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"), T,
                                      _ptr(counts, torch.int32, "counts"), _ptr(offsets, torch.int32, "offsets"),
                                      _ptr(gather_idx, torch.int32, "gather_idx"),
                                      _ptr(scatter_idx, torch.int32, "scatter_idx"), _stream(stream)),
           "moe_permute_noalloc")
    return counts, offsets, gather_idx, scatter_idx


def moe_grouped_swiglu(cfg, weights: DeviceWeights, x_routed, gather_idx, offsets, ws, y=None, stream=None):
    T = x_routed.shape[0]
    Lr = x_routed.shape[1]
    rows = moe_permuted_rows(cfg, T)
    y = torch.empty((max(rows, 1), Lr), dtype=torch.bfloat16, device=x_routed.device) if y is None else y
    ws_ = weights.struct()
    _check(load().moe_grouped_swiglu(ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x_routed, torch.bfloat16, "x_routed"),
                                     _ptr(gather_idx, torch.int32, "gather_idx"), _ptr(offsets, torch.int32, "offsets"),
                                     T, _ptr(y, torch.bfloat16, "y"), _ptr(ws, None, "ws"), ws.numel(),
                                     _stream(stream)), "moe_grouped_swiglu")
    return y


def moe_grouped_swiglu_preact(cfg, weights: DeviceWeights, x_routed, gather_idx, offsets, ws, y=None, preact=None,
                              stream=None):
    """moe_grouped_swiglu that also returns the pre-activations [u | g] ((rows, 2h) bf16)."""
    T = x_routed.shape[0]
    Lr = x_routed.shape[1]
    rows = moe_permuted_rows(cfg, T)
    dev = x_routed.device
    y = torch.empty((max(rows, 1), Lr), dtype=torch.bfloat16, device=dev) if y is None else y
    preact = (torch.empty((max(rows, 1), 2 * cfg.hidden_size), dtype=torch.bfloat16, device=dev)
              if preact is None else preact)
    ws_ = weights.struct()
    _check(load().moe_grouped_swiglu_preact(
        ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x_routed, torch.bfloat16, "x_routed"),
        _ptr(gather_idx, torch.int32, "gather_idx"), _ptr(offsets, torch.int32, "offsets"), T,
        _ptr(y, torch.bfloat16, "y"), _ptr(preact, torch.bfloat16, "preact"), _ptr(ws, None, "ws"), ws.numel(),
        _stream(stream)), "moe_grouped_swiglu_preact")
    return y, preact


def moe_combine(cfg, y, scatter_idx, w, T, z=None, stream=None):
    Lr = y.shape[1]
    z = torch.empty((T, Lr), dtype=torch.bfloat16, device=y.device) if z is None else z
    _check(load().moe_combine(ctypes.byref(cfg), _ptr(y, torch.bfloat16, "y"), _ptr(scatter_idx, torch.int32, "scatter_idx"),
                              _ptr(w, torch.float32, "weights"), T, _ptr(z, torch.bfloat16, "z"), _stream(stream)),
           "moe_combine")
    return z


def moe_latent_down(cfg, weights: DeviceWeights, x, ws, x_routed=None, stream=None):
    T = x.shape[0]
    x_routed = torch.empty((T, cfg.latent_dim), dtype=torch.bfloat16, device=x.device) if x_routed is None else x_routed
    ws_ = weights.struct()
    _check(load().moe_latent_down(ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x, torch.bfloat16, "x"), T,
                                  _ptr(x_routed, torch.bfloat16, "x_routed"), _ptr(ws, None, "ws"), ws.numel(),
                                  _stream(stream)), "moe_latent_down")
    return x_routed


def moe_latent_restore(cfg, weights: DeviceWeights, z, ws, out=None, stream=None):
    T = z.shape[0]
    out = torch.empty((T, cfg.d_model), dtype=torch.bfloat16, device=z.device) if out is None else out
    ws_ = weights.struct()
    _check(load().moe_latent_restore(ctypes.byref(cfg), ctypes.byref(ws_), _ptr(z, torch.bfloat16, "z"), T,
                                     _ptr(out, torch.bfloat16, "out"), _ptr(ws, None, "ws"), ws.numel(),
                                     _stream(stream)), "moe_latent_restore")
    return out


def moe_layer_forward(cfg, weights: DeviceWeights, x, ws, out=None, stream=None):
    T = x.shape[0]
    out = torch.empty((T, cfg.d_model), dtype=torch.bfloat16, device=x.device) if out is None else out
    ws_ = weights.struct()
    _check(load().moe_layer_forward(ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x, torch.bfloat16, "x"), T,
                                    _ptr(out, torch.bfloat16, "out"), _ptr(ws, None, "ws"), ws.numel(),
                                    _stream(stream)), "moe_layer_forward")
    return out


def moe_layer_forward_preact(cfg, weights: DeviceWeights, x, ws, out=None, preact=None, logits=None, stream=None):
    """The layer forward that keeps the experts' pre-activations: (out, preact (rows, 2h) bf16).
    logits (optional (T, E) fp32 tensor) also receives the router logits."""
    T = x.shape[0]
    out = torch.empty((T, cfg.d_model), dtype=torch.bfloat16, device=x.device) if out is None else out
    rows = moe_permuted_rows(cfg, T)
    preact = (torch.empty((max(rows, 1), 2 * cfg.hidden_size), dtype=torch.bfloat16, device=x.device)
              if preact is None else preact)
    ws_ = weights.struct()
    _check(load().moe_layer_forward_preact(ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x, torch.bfloat16, "x"), T,
                                           _ptr(out, torch.bfloat16, "out"), _ptr(preact, torch.bfloat16, "preact"),
                                           None if logits is None else _ptr(logits, torch.float32, "logits"),
                                           _ptr(ws, None, "ws"), ws.numel(), _stream(stream)),
           "moe_layer_forward_preact")
    return out, preact


def _host_ptr(t: torch.Tensor, name: str) -> int:
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if not t.is_contiguous() or t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be a contiguous bf16 tensor")
    return t.data_ptr()


def host_workspace(cfg: moe_config_t, T: int, device="cuda") -> torch.Tensor:
    """A device workspace of moe_host_workspace_size bytes."""
    n = ctypes.c_size_t()
    _check(load().moe_host_workspace_size(ctypes.byref(cfg), T, ctypes.byref(n)), "moe_host_workspace_size")
    return torch.empty(max(1, n.value), dtype=torch.uint8, device=device)


def moe_layer_forward_host_batches(cfg, weights: DeviceWeights, x_hosts, out_hosts, ws, stream=None):
    """The layer over host batches (lists of host (T, d_model) bf16 tensors, pinned for asynchronous
    copies); outputs are complete once the stream is."""
    if len(x_hosts) != len(out_hosts) or not x_hosts:
        raise ValueError("x_hosts and out_hosts must be non-empty lists of the same length")
    T = x_hosts[0].shape[0]
    for x, o in zip(x_hosts, out_hosts):
        if tuple(x.shape) != (T, cfg.d_model) or tuple(o.shape) != (T, cfg.d_model):
            raise ValueError("every batch must be (T, d_model)")
    n = len(x_hosts)
    xs = (ctypes.c_void_p * n)(*[_host_ptr(x, "x_host") for x in x_hosts])
    os_ = (ctypes.c_void_p * n)(*[_host_ptr(o, "out_host") for o in out_hosts])
    ws_ = weights.struct()
    _check(load().moe_layer_forward_host_batches(ctypes.byref(cfg), ctypes.byref(ws_), xs, os_, n, T,
                                                 _ptr(ws, None, "ws"), ws.numel(), _stream(stream)),
           "moe_layer_forward_host_batches")
    return out_hosts


STAGES = ["latent_down", "router_gemm", "topk", "permute", "gather", "grouped_gemm1_swiglu",
          "grouped_gemm2", "combine", "latent_up"]


def moe_layer_forward_staged(cfg, weights: DeviceWeights, x, ws, events, out=None, stream=None):
    """moe_layer_forward recording 10 torch.cuda.Event objects at the stage boundaries."""
    T = x.shape[0]
    out = torch.empty((T, cfg.d_model), dtype=torch.bfloat16, device=x.device) if out is None else out
    handles = (ctypes.c_void_p * 10)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    ws_ = weights.struct()
    _check(load().moe_layer_forward_staged(ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x, torch.bfloat16, "x"), T,
                                           _ptr(out, torch.bfloat16, "out"), _ptr(ws, None, "ws"), ws.numel(),
                                           _stream(stream), handles), "moe_layer_forward_staged")
    return out


def moe_layer_forward_launches(cfg, T: int) -> int:
    n = ctypes.c_int32()
    _check(load().moe_layer_forward_launches(ctypes.byref(cfg), T, ctypes.byref(n)), "moe_layer_forward_launches")
    return n.value


def moe_backward_workspace_size(cfg: moe_config_t, T: int) -> int:
    out = ctypes.c_size_t()
    _check(load().moe_backward_workspace_size(ctypes.byref(cfg), T, ctypes.byref(out)), "moe_backward_workspace_size")
    return out.value


def backward_workspace(cfg, T, device="cuda") -> torch.Tensor:
    return torch.empty(max(1, moe_backward_workspace_size(cfg, T)), dtype=torch.uint8, device=device)


def moe_combine_backward(cfg, dz, y, scatter_idx, weights, gather_idx=None, dy=None, dweights=None, stream=None):
    """dy (rows, L') bf16 and dweights (T, k) fp32 of the weighted combine."""
    T = dz.shape[0]
    dy = torch.empty_like(y) if dy is None else dy
    dweights = torch.empty((T, cfg.top_k), dtype=torch.float32, device=dz.device) if dweights is None else dweights
    _check(load().moe_combine_backward(ctypes.byref(cfg), _ptr(dz, torch.bfloat16, "dz"), _ptr(y, torch.bfloat16, "y"),
                                       _ptr(scatter_idx, torch.int32, "scatter_idx"),
                                       _ptr(gather_idx, torch.int32, "gather_idx"), _ptr(weights, torch.float32, "weights"),
                                       T, _ptr(dy, torch.bfloat16, "dy"), _ptr(dweights, torch.float32, "dweights"),
                                       _stream(stream)), "moe_combine_backward")
    return dy, dweights


def moe_grouped_swiglu_backward(cfg, weights: DeviceWeights, x_routed, gather_idx, offsets, scatter_idx, dy, bws,
                                dx_routed=None, dw_up_gate=None, dw_out=None, stream=None):
    """Input and weight gradients of the grouped SwiGLU experts (bws: backward_workspace)."""
    T, Lr = x_routed.shape
    E, h = cfg.num_experts, cfg.hidden_size
    dev = x_routed.device
    dx_routed = torch.empty((T, Lr), dtype=torch.bfloat16, device=dev) if dx_routed is None else dx_routed
    dw_up_gate = torch.empty((E, 2 * h, Lr), dtype=torch.float32, device=dev) if dw_up_gate is None else dw_up_gate
    dw_out = torch.empty((E, Lr, h), dtype=torch.float32, device=dev) if dw_out is None else dw_out
    ws_ = weights.struct()
    _check(load().moe_grouped_swiglu_backward(
        ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x_routed, torch.bfloat16, "x_routed"),
        _ptr(gather_idx, torch.int32, "gather_idx"), _ptr(offsets, torch.int32, "offsets"),
        _ptr(scatter_idx, torch.int32, "scatter_idx"), T, _ptr(dy, torch.bfloat16, "dy"),
        _ptr(dx_routed, torch.bfloat16, "dx_routed"), _ptr(dw_up_gate, torch.float32, "dw_up_gate"),
        _ptr(dw_out, torch.float32, "dw_out"), _ptr(bws, None, "ws"), bws.numel(), _stream(stream)),
        "moe_grouped_swiglu_backward")
    return dx_routed, dw_up_gate, dw_out


def moe_grouped_swiglu_backward_preact(cfg, weights: DeviceWeights, x_routed, gather_idx, offsets, scatter_idx, dy,
                                       preact, bws, dx_routed=None, dw_up_gate=None, dw_out=None, stream=None):
    """moe_grouped_swiglu_backward from the forward's saved pre-activations (preact (rows, 2h) bf16)."""
    T, Lr = x_routed.shape
    E, h = cfg.num_experts, cfg.hidden_size
    dev = x_routed.device
    dx_routed = torch.empty((T, Lr), dtype=torch.bfloat16, device=dev) if dx_routed is None else dx_routed
    dw_up_gate = torch.empty((E, 2 * h, Lr), dtype=torch.float32, device=dev) if dw_up_gate is None else dw_up_gate
    dw_out = torch.empty((E, Lr, h), dtype=torch.float32, device=dev) if dw_out is None else dw_out
    ws_ = weights.struct()
    _check(load().moe_grouped_swiglu_backward_preact(
        ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x_routed, torch.bfloat16, "x_routed"),
        _ptr(gather_idx, torch.int32, "gather_idx"), _ptr(offsets, torch.int32, "offsets"),
        _ptr(scatter_idx, torch.int32, "scatter_idx"), T, _ptr(dy, torch.bfloat16, "dy"),
        _ptr(preact, torch.bfloat16, "preact"), _ptr(dx_routed, torch.bfloat16, "dx_routed"),
        _ptr(dw_up_gate, torch.float32, "dw_up_gate"), _ptr(dw_out, torch.float32, "dw_out"),
        _ptr(bws, None, "ws"), bws.numel(), _stream(stream)), "moe_grouped_swiglu_backward_preact")
    return dx_routed, dw_up_gate, dw_out


def moe_latent_restore_backward(cfg, weights: DeviceWeights, z, dout, bws, stream=None):
    """(dz (T, L) bf16, dw_up (D, L) fp32, drms_weight (L,) fp32 or None without the norm)."""
    T, L = z.shape
    D = cfg.d_model
    dev = z.device
    dz = torch.empty((T, L), dtype=torch.bfloat16, device=dev)
    dw_up = torch.empty((D, L), dtype=torch.float32, device=dev)
    dg = torch.empty(L, dtype=torch.float32, device=dev) if cfg.up_proj_norm else None
    ws_ = weights.struct()
    _check(load().moe_latent_restore_backward(
        ctypes.byref(cfg), ctypes.byref(ws_), _ptr(z, torch.bfloat16, "z"), T, _ptr(dout, torch.bfloat16, "dout"),
        _ptr(dz, torch.bfloat16, "dz"), _ptr(dw_up, torch.float32, "dw_up"),
        None if dg is None else _ptr(dg, torch.float32, "drms_weight"), _ptr(bws, None, "ws"), bws.numel(),
        _stream(stream)), "moe_latent_restore_backward")
    return dz, dw_up, dg


def moe_latent_down_backward(cfg, weights: DeviceWeights, x, dx_routed, bws, stream=None):
    """(dx (T, D) bf16, dw_down (L, D) fp32)."""
    T, D = x.shape
    L = cfg.latent_dim
    dev = x.device
    dx = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    dw_down = torch.empty((L, D), dtype=torch.float32, device=dev)
    ws_ = weights.struct()
    _check(load().moe_latent_down_backward(
        ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x, torch.bfloat16, "x"), T,
        _ptr(dx_routed, torch.bfloat16, "dx_routed"), _ptr(dx, torch.bfloat16, "dx"),
        _ptr(dw_down, torch.float32, "dw_down"), _ptr(bws, None, "ws"), bws.numel(), _stream(stream)),
        "moe_latent_down_backward")
    return dx, dw_down


def mx_scale_ld(cols: int) -> int:
    """Bytes per row of MXFP8 block scales: cols / 32, rounded up to 16."""
    return (cols // 32 + 15) // 16 * 16


def moe_quantize_mxfp8(x, stream=None):
    """(codes (rows, cols) uint8 e4m3 bits, scales (rows, mx_scale_ld(cols)) uint8 E8M0 exponents)."""
    rows, cols = x.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    scales = torch.zeros((rows, mx_scale_ld(cols)), dtype=torch.uint8, device=x.device)
    _check(load().moe_quantize_mxfp8(_ptr(x, torch.bfloat16, "x"), rows, cols, _ptr(codes, torch.uint8, "codes"),
                                     _ptr(scales, torch.uint8, "scales"), scales.shape[1], _stream(stream)),
           "moe_quantize_mxfp8")
    return codes, scales


def moe_check_wait_timeout(limit_ms: int = 20, stream=None) -> int:
    """Runs a bounded wait that nothing completes; returns how many ms it waited before giving up
    (raises if the timeout was not reported through the status word)."""
    waited = ctypes.c_int32()
    _check(load().moe_check_wait_timeout(limit_ms, ctypes.byref(waited), _stream(stream)), "moe_check_wait_timeout")
    return waited.value


def layer_backward_workspace(cfg, T, device="cuda") -> torch.Tensor:
    n = ctypes.c_size_t()
    _check(load().moe_layer_backward_workspace_size(ctypes.byref(cfg), T, ctypes.byref(n)),
           "moe_layer_backward_workspace_size")
    return torch.empty(max(1, n.value), dtype=torch.uint8, device=device)


def moe_layer_backward(cfg, weights: DeviceWeights, x, ws, preact, logits, dout, bws, dx=None, stream=None):
    """The whole layer's backward after moe_layer_forward_preact(x, ws): (dx (T, D) bf16, a dict of the
    fp32 weight gradients: dw_router, db_router, dw_up_gate, dw_out and, when latent, dw_down_latent,
    dw_up_latent, drms_weight; entries the configuration has no weight for are None)."""
    T, D = x.shape
    E, h = cfg.num_experts, cfg.hidden_size
    Lr = cfg.latent_dim or cfg.d_model
    dev = x.device
    f32 = lambda *shape: torch.empty(shape, dtype=torch.float32, device=dev)   # noqa: E731
    grads = {"dw_router": f32(E, D), "db_router": f32(E) if cfg.router_bias else None,
             "dw_up_gate": f32(E, 2 * h, Lr), "dw_out": f32(E, Lr, h),
             "dw_down_latent": f32(Lr, D) if cfg.latent_dim else None,
             "dw_up_latent": f32(D, Lr) if cfg.latent_dim else None,
             "drms_weight": f32(Lr) if cfg.latent_dim and cfg.up_proj_norm else None}
    g = moe_grads_t(*[None if grads[n] is None else _ptr(grads[n], torch.float32, n)
                      for n, _ in moe_grads_t._fields_])
    dx = torch.empty((T, D), dtype=torch.bfloat16, device=dev) if dx is None else dx
    ws_ = weights.struct()
    _check(load().moe_layer_backward(
        ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x, torch.bfloat16, "x"), T, _ptr(ws, None, "ws"), ws.numel(),
        None if preact is None else _ptr(preact, torch.bfloat16, "preact"), _ptr(logits, torch.float32, "logits"),
        _ptr(dout, torch.bfloat16, "dout"), _ptr(dx, torch.bfloat16, "dx"), ctypes.byref(g), _ptr(bws, None, "bws"),
        bws.numel(), _stream(stream)), "moe_layer_backward")
    return dx, grads


def moe_router_backward(cfg, weights: DeviceWeights, x, logits, idx, dweights, bws, stream=None):
    """(dlogits (T,E) fp32, dx (T,D) bf16, dw_router (E,D) fp32, db_router (E,) fp32 or None)."""
    T, D = x.shape
    E = cfg.num_experts
    dev = x.device
    dlogits = torch.empty((T, E), dtype=torch.float32, device=dev)
    dx = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((E, D), dtype=torch.float32, device=dev)
    db = torch.empty(E, dtype=torch.float32, device=dev) if cfg.router_bias else None
    ws_ = weights.struct()
    _check(load().moe_router_backward(
        ctypes.byref(cfg), ctypes.byref(ws_), _ptr(x, torch.bfloat16, "x"), T, _ptr(logits, torch.float32, "logits"),
        _ptr(idx, torch.int32, "idx"), _ptr(dweights, torch.float32, "dweights"), _ptr(dlogits, torch.float32, "dlogits"),
        _ptr(dx, torch.bfloat16, "dx"), _ptr(dw, torch.float32, "dw_router"), _ptr(db, torch.float32, "db_router"),
        _ptr(bws, None, "ws"), bws.numel(), _stream(stream)), "moe_router_backward")
    return dlogits, dx, dw, db


def moe_accumulate_counts(counts, accum, stream=None):
    """accum (E, int64) += counts (E, int32), on the device."""
    _check(load().moe_accumulate_counts(_ptr(counts, torch.int32, "counts"), counts.numel(),
                                        _ptr(accum, torch.int64, "accum"), _stream(stream)), "moe_accumulate_counts")
    return accum


def moe_load_imbalance(counts, out=None, stream=None):
    """max / mean of a per-expert counter (int32 or int64), as a device float scalar."""
    out = torch.empty(1, dtype=torch.float32, device=counts.device) if out is None else out
    if counts.dtype not in (torch.int32, torch.int64):
        raise ValueError("counts must be int32 or int64")
    _check(load().moe_load_imbalance(_ptr(counts, None, "counts"), int(counts.dtype == torch.int64), counts.numel(),
                                     _ptr(out, torch.float32, "imbalance"), _stream(stream)), "moe_load_imbalance")
    return out


def moe_score_bias_update(accum, bias_gamma: float, score_bias, stream=None):
    """score_bias += gamma * sign(mean(accum) - accum); accum = 0 (both in place, on the device)."""
    _check(load().moe_score_bias_update(_ptr(accum, torch.int64, "accum"), accum.numel(), bias_gamma,
                                        _ptr(score_bias, torch.float32, "score_bias"), _stream(stream)),
           "moe_score_bias_update")
    return score_bias


def moe_get_status(stream=None, clear: bool = True) -> int:
    """Synchronises the stream and returns (and by default clears) the device status word."""
    out = ctypes.c_int32()
    _check(load().moe_get_status(_stream(stream), ctypes.byref(out), int(clear)), "moe_get_status")
    return out.value


def layer_intermediates(cfg, T, ws):
    """Views into the workspace of the layer forward's intermediates (after moe_layer_forward)."""
    o = moe_workspace_layout(cfg, T)
    E, k = cfg.num_experts, cfg.top_k
    Lr = cfg.latent_dim or cfg.d_model
    R = T * k
    rows = moe_permuted_rows(cfg, T)

    def view(off, n, dtype, shape):
        size = torch.tensor([], dtype=dtype).element_size()
        return ws[off:off + n * size].view(dtype).view(*shape)

    out = {
        # y: the training forward's bf16 rows; after moe_layer_forward of a configuration that keeps
        # them in fp32 (moe_layer_expert_rows_fp32), "y_f32" holds them
        "idx": view(o[1], R, torch.int32, (T, k)),
        "weights": view(o[2], R, torch.float32, (T, k)),
        "counts": view(o[3], E, torch.int32, (E,)),
        "offsets": view(o[4], E + 1, torch.int32, (E + 1,)),
        "gather_idx": view(o[5], rows, torch.int32, (rows,)),
        "scatter_idx": view(o[6], R, torch.int32, (R,)),
        "y": view(o[8], rows * Lr, torch.bfloat16, (rows, Lr)),
    }
    if moe_layer_expert_rows_fp32(cfg):
        out["y_f32"] = view(o[8], rows * Lr, torch.float32, (rows, Lr))
    if o[7] >= 0:
        out["x_routed"] = view(o[7], T * cfg.latent_dim, torch.bfloat16, (T, cfg.latent_dim))
    if o[9] >= 0:
        out["z_normalised"] = view(o[9], T * cfg.latent_dim, torch.bfloat16, (T, cfg.latent_dim))
    return out
