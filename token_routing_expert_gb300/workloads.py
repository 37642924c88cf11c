"""Seeded synthetic workloads for the MoE layer forward.

This module only draws inputs.  It holds none of the layer's arithmetic; the
CUDA path (through the C-ABI) and the float64 oracle both consume exactly the
bf16 / fp32 tensors it returns.

Recipe (every tensor has its own counter-free stream, so any expert's weights
can be redrawn alone and the draw does not depend on the thread count):

  stream (seed, 0)      x            (T, d_model)          N(0, 1)     -> bf16
  stream (seed, 1)      w_router     (E, d_model)          N(0, 0.02)  -> bf16
  stream (seed, 2)      expert rank permutation (skewed load only)
  stream (seed, 3)      score_bias   (E,)                  N(0, std)   fp32
  stream (seed, 4)      w_down       (L, d_model)          N(0, 0.02)  -> bf16
  stream (seed, 5)      w_up_latent  (d_model, L)          N(0, 0.02)  -> bf16
  stream (seed, 6, e)   w_up_gate[e] (2h, L)  rows [0,h) up, [h,2h) gate, N(0, 0.02) -> bf16
  stream (seed, 7, e)   w_out[e]     (L, h)                N(0, 0.02)  -> bf16

Each stream is numpy ``PCG64(SeedSequence([seed, stream(, e)]))`` drawing
float32 standard normals, scaled, then rounded to bf16 (round to nearest
even, by torch's conversion).  The skewed load of the latent prefill workload
adds a router bias b[e] = 0.5 * ln(1 / rank_e), rank_e = 1 + the position of
expert e in a seeded permutation of the experts.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from typing import Dict, Optional

import numpy as np
import torch

GATING_NAMES = {"softmax": 0, "topk_softmax": 1, "sigmoid": 2}


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    T: int
    d_model: int
    num_experts: int
    top_k: int
    hidden_size: int
    latent_dim: int = 0
    gating: str = "softmax"
    sigmoid_stability_epsilon: float = 0.0
    normalize_expert_weights: float = 0.0
    restore_weight_scale: bool = False
    expert_weight_scale: float = 0.0
    original_top_k: int = 0
    score_bias_std: float = 0.0          # > 0: draw a selection-only score bias
    skew: bool = False                   # per-expert logit offset 0.5*ln(1/rank)
    up_proj_norm: bool = True
    rms_eps: float = 1e-6
    capacity_factor: float = 0.0         # > 0: capacity-limited experts
    expert_fp8: int = 0                  # experts' operands: 0 bf16, 1 rowwise e4m3, 2 MXFP8
    x_std: float = 1.0
    w_std: float = 0.02
    seed: int = 0

    @property
    def routed_dim(self) -> int:
        return self.latent_dim if self.latent_dim else self.d_model

    @property
    def rows(self) -> int:
        return self.T * self.top_k

    def with_(self, **kw) -> "WorkloadSpec":
        return replace(self, **kw)


# The five workloads: a tiny one, an OlmoE-shaped one, a sigmoid-gated wide
# one, a skewed latent ultra-sparse prefill and a latent decode batch.
WORKLOADS: Dict[str, WorkloadSpec] = {
    "tiny": WorkloadSpec("tiny", T=256, d_model=256, num_experts=8, top_k=2, hidden_size=128,
                         gating="softmax", normalize_expert_weights=1.0, seed=0),
    "olmoe": WorkloadSpec("olmoe", T=8192, d_model=2048, num_experts=64, top_k=8, hidden_size=1024,
                          gating="topk_softmax", seed=1),
    "sigmoid_wide": WorkloadSpec("sigmoid_wide", T=16384, d_model=4096, num_experts=256, top_k=8,
                                 hidden_size=2048, gating="sigmoid", sigmoid_stability_epsilon=1e-6,
                                 score_bias_std=0.01, normalize_expert_weights=1.0,
                                 restore_weight_scale=True, seed=2),
    "latent_prefill": WorkloadSpec("latent_prefill", T=32768, d_model=7168, num_experts=896, top_k=8,
                                   hidden_size=1024, latent_dim=2048, gating="sigmoid", skew=True, seed=3),
    "latent_decode": WorkloadSpec("latent_decode", T=64, d_model=7168, num_experts=896, top_k=8,
                                  hidden_size=1024, latent_dim=2048, gating="sigmoid", seed=4),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _normal_bf16(shape, std: float, *key: int) -> torch.Tensor:
    a = _rng(*key).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).to(torch.bfloat16)


def expert_weights(spec: WorkloadSpec, e: int):
    """Expert e's (w_up_gate (2h, L), w_out (L, h)) as bf16, drawn alone."""
    h, L = spec.hidden_size, spec.routed_dim
    return (_normal_bf16((2 * h, L), spec.w_std, spec.seed, 6, e),
            _normal_bf16((L, h), spec.w_std, spec.seed, 7, e))


def skew_bias(spec: WorkloadSpec) -> np.ndarray:
    """Per-expert logit offset 0.5 * ln(1 / rank) over a seeded expert permutation (fp32)."""
    perm = _rng(spec.seed, 2).permutation(spec.num_experts)
    rank = np.empty(spec.num_experts, np.int64)
    rank[perm] = np.arange(1, spec.num_experts + 1)
    return (0.5 * np.log(1.0 / rank.astype(np.float64))).astype(np.float32)


def generate(spec: WorkloadSpec, threads: Optional[int] = None, experts: bool = True) -> Dict[str, torch.Tensor]:
    """Draw every input of the workload as CPU tensors.

    Keys: x, w_router, b_router (fp32 or None), score_bias (fp32 or None),
    w_down, w_up_latent (None unless latent), w_up_gate (E, 2h, L),
    w_out (E, L, h).  ``experts=False`` skips the expert weights.
    """
    T, D, E, h, L = spec.T, spec.d_model, spec.num_experts, spec.hidden_size, spec.routed_dim
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["x"] = _normal_bf16((T, D), spec.x_std, spec.seed, 0)
    out["w_router"] = _normal_bf16((E, D), spec.w_std, spec.seed, 1)
    out["b_router"] = torch.from_numpy(skew_bias(spec)) if spec.skew else None
    if spec.score_bias_std > 0:
        sb = _rng(spec.seed, 3).standard_normal(E, dtype=np.float32) * np.float32(spec.score_bias_std)
        out["score_bias"] = torch.from_numpy(sb)
    else:
        out["score_bias"] = None
    if spec.latent_dim:
        out["w_down"] = _normal_bf16((L, D), spec.w_std, spec.seed, 4)
        out["w_up_latent"] = _normal_bf16((D, L), spec.w_std, spec.seed, 5)
    else:
        out["w_down"] = None
        out["w_up_latent"] = None
    if experts:
        w_ug = torch.empty((E, 2 * h, L), dtype=torch.bfloat16)
        w_o = torch.empty((E, L, h), dtype=torch.bfloat16)

        def fill(e: int) -> None:
            a, b = expert_weights(spec, e)
            w_ug[e].copy_(a)
            w_o[e].copy_(b)

        n = threads or min(32, os.cpu_count() or 1)
        if n <= 1 or E == 1:
            for e in range(E):
                fill(e)
        else:
            with ThreadPoolExecutor(n) as ex:
                list(ex.map(fill, range(E)))
        out["w_up_gate"] = w_ug
        out["w_out"] = w_o
    return out


def algorithmic_flops(spec: WorkloadSpec) -> int:
    """GEMM FLOPs of one forward (2 per multiply-add): router + latent projections + active experts."""
    f = 2 * spec.T * spec.d_model * spec.num_experts
    if spec.latent_dim:
        f += 4 * spec.T * spec.d_model * spec.latent_dim
    f += 6 * spec.routed_dim * spec.hidden_size * spec.rows
    return f


def algorithmic_bytes(spec: WorkloadSpec, experts_touched: int) -> int:
    """Touched expert weights + router weights + latent weights + x in + out (bf16)."""
    b = experts_touched * 3 * spec.routed_dim * spec.hidden_size * 2
    b += spec.num_experts * spec.d_model * 2
    if spec.latent_dim:
        b += 2 * spec.d_model * spec.latent_dim * 2
    b += 2 * spec.T * spec.d_model * 2
    return b
