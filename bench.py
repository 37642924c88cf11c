#!/usr/bin/env python3
"""Benchmark of the MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl native|reference]

A step is one moe_layer_forward (latent down-projection, router GEMM, top-k,
permutation, grouped SwiGLU GEMMs, combine, RMSNorm + up-projection) over
one batch of T synthetic tokens resident in HBM.  The default workload is
the largest one, the skewed latent ultra-sparse prefill (T=32768,
d_model=7168, latent_dim=2048, 896 experts, top-8, hidden 1024, sigmoid
gating), which runs every step of the path.  The same invocation also times
the latent decode batch (T=64, the same layer shape, bound by HBM) and
reports it in the line's ``decode`` object.  With N > 1 (torchrun), every rank runs its own
replica on its own batch: tokens are independent, so there is no collective
on the data path (weak scaling); the barrier and the max over ranks are the
only communication.

``--impl reference`` times the float64 CPU oracle, as it stands, on a
bounded sample of the same workload on the host cores (rank 0 only).

Prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from token_routing_expert_gb300 import workloads as W  # noqa: E402

METRIC = "MoE layer fwd tokens/s and TFLOP/s (frac of bf16 peak); decode GB/s vs HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(spec: W.WorkloadSpec) -> str:
    """One-line description of the workload."""
    s = (f"{spec.name}: T={spec.T} d_model={spec.d_model} experts={spec.num_experts} top_k={spec.top_k} "
         f"hidden={spec.hidden_size} gating={spec.gating}")
    if spec.latent_dim:
        s += f" latent_dim={spec.latent_dim} rmsnorm"
    if spec.score_bias_std:
        s += f" score_bias~N(0,{spec.score_bias_std})"
    if spec.normalize_expert_weights:
        s += f" p={spec.normalize_expert_weights:g}"
    if spec.restore_weight_scale:
        s += " restore_weight_scale"
    if spec.skew:
        s += " skewed_load"
    if spec.capacity_factor:
        s += f" capacity_factor={spec.capacity_factor:g}"
    if spec.expert_fp8 == 2:
        s += " experts_mxfp8"
    elif spec.expert_fp8:
        s += " experts_e4m3_rowwise"
    return s


class ClockSampler:
    """nvidia-smi clock / throttle samples every 20 ms; keeps the samples inside [t0, t1]."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.02 <= r[0] <= t1 + 0.02]
        window = "timed region"
        if not inside:  # region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: abs(r[0] - 0.5 * (t0 + t1)))[:3]
            window = "nearest samples to a short timed region"
        reasons = sorted({self.REASONS[i] for r in inside for i in range(4) if r[3][i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(inside), "window": window}


def bench_config(spec: W.WorkloadSpec, world: int) -> dict:
    """The `config` object of the JSON line (identical keys in both arms)."""
    return {"workload": workload_desc(spec), "T_per_gpu": spec.T, "global_tokens": world * spec.T,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def rank_inputs(spec: W.WorkloadSpec, rank: int, experts: bool = True):
    """Inputs of one replica: shared weights, and a batch of tokens of the rank's own."""
    inp = W.generate(spec, experts=experts)
    if rank > 0:
        inp["x"] = W.generate(spec.with_(seed=spec.seed * 1000 + rank), experts=False)["x"]
    return inp


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's value (the job's time); identity without a process group."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job throughput: all ranks' tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def kernel_traffic(workload: str):
    """Per-launch DRAM bytes of the grouped SwiGLU GEMM from the committed ncu summary,
    if the kernel source has not changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"grouped_gemm1_swiglu_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    src = os.path.join(ROOT, "token_routing_expert_gb300", "csrc", "gemm_tc.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if vals.get("gemm_tc_cu_sha256") != digest or "dram_bytes_per_launch" not in vals:
        return None
    return float(vals["dram_bytes_per_launch"])


def oracle_sample_rate(spec: W.WorkloadSpec, inp, n_tokens: int, min_seconds: float, max_reps: int = 50):
    """Times the float64 oracle on the first n_tokens tokens; returns (tokens/s, reps, seconds)."""
    from oracle import moe_ref as ref  # the CPU baseline leg is the only user of the oracle here

    h = spec.hidden_size

    def f64(t):
        return None if t is None else t.to(torch.float64).numpy()

    cfg = ref.OracleConfig(d_model=spec.d_model, num_experts=spec.num_experts, top_k=spec.top_k, hidden_size=h,
                           latent_dim=spec.latent_dim, up_proj_norm=spec.up_proj_norm, rms_eps=spec.rms_eps,
                           gating=W.GATING_NAMES[spec.gating],
                           sigmoid_stability_epsilon=spec.sigmoid_stability_epsilon,
                           normalize_expert_weights=spec.normalize_expert_weights,
                           restore_weight_scale=spec.restore_weight_scale,
                           expert_weight_scale=spec.expert_weight_scale, original_top_k=spec.original_top_k,
                           router_bias=spec.skew, has_score_bias=spec.score_bias_std > 0)
    wug, wo = inp["w_up_gate"], inp["w_out"]
    wts = ref.OracleWeights(w_router=f64(inp["w_router"]),
                            expert=lambda e: (f64(wug[e][:h]), f64(wug[e][h:]), f64(wo[e])),
                            b_router=f64(inp["b_router"]), score_bias=f64(inp["score_bias"]),
                            w_down_latent=f64(inp["w_down"]), w_up_latent=f64(inp["w_up_latent"]))
    x = f64(inp["x"][:n_tokens])
    t0 = time.perf_counter()
    reps = 0
    while True:
        ref.layer_forward(cfg, x, wts)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return n_tokens * reps / el, reps, el


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    spec = W.WORKLOADS[args.config]
    inp = W.generate(spec)
    # each step is a bounded sample: as many tokens (up to --ref-tokens) as keep the K timed
    # steps near --ref-seconds, from the rate of a short calibration call
    probe = min(spec.T, 8)
    rate, _, _ = oracle_sample_rate(spec, inp, probe, 0.0, max_reps=1)
    n = int(max(1, min(spec.T, args.ref_tokens, rate * args.ref_seconds / max(args.steps, 1))))
    for _ in range(args.warmup):
        oracle_sample_rate(spec, inp, n, 0.0, max_reps=1)
    rates = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        r, _, _ = oracle_sample_rate(spec, inp, n, 0.0, max_reps=1)
        rates.append(r)
    el = time.perf_counter() - t_all
    value = n * args.steps / el
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(spec, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {spec.T} tokens per step, full layer in float64 numpy"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def decode_pass(args, native, name, peaks, dist):
    """Times the decode-shaped workload (bound by HBM) in the same invocation: K plain forwards,
    CUDA events on the launching stream; returns the line's ``decode`` object."""
    spec = W.WORKLOADS[name]
    inp = W.generate(spec)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    x = inp["x"].cuda()
    ws = native.workspace(cfg, spec.T)
    out = torch.empty((spec.T, spec.d_model), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 1)):
        native.moe_layer_forward(cfg, wts, x, ws, out=out)
    torch.cuda.synchronize()
    if native.moe_get_status() != 0:
        raise SystemExit("device status error in the decode warm-up")
    touched = int((native.layer_intermediates(cfg, spec.T, ws)["counts"] > 0).sum().item())
    alg_bytes = W.algorithmic_bytes(spec, touched)
    L2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    flush = alg_bytes < 2 * L2
    flush_buf = torch.empty(2 * L2 // 4 + 1024, dtype=torch.float32, device="cuda") if flush else None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        if flush:
            flush_buf.fill_(float(i))
        ev[i][0].record(stream)
        native.moe_layer_forward(cfg, wts, x, ws, out=out)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if native.moe_get_status() != 0:
        raise SystemExit("device status error in the decode pass")
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / args.steps, dist, "cuda")
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    flops = W.algorithmic_flops(spec)
    roof_ms = 1e3 * max(alg_bytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    del wts, ws, x, out, flush_buf
    torch.cuda.empty_cache()
    return {"workload": workload_desc(spec), "ms_per_step": ms, "tokens_per_s": spec.T / (ms * 1e-3),
            "gbs": gbs, "hbm_peak": peaks["hbm_gbs"], "frac_hbm_peak": gbs / peaks["hbm_gbs"],
            "bound": "hbm", "roofline_ms": roof_ms, "frac_of_roofline": roof_ms / ms,
            "experts_touched": touched, "algorithmic_bytes": alg_bytes, "algorithmic_flops": flops,
            "steps": args.steps, "l2": "flushed between steps" if flush else "no flush (bytes per step > 2x L2)",
            "note": "algorithmic bytes = touched expert weights + router + latent weights + x + out, each once; "
                    "events around each forward"}


def run_native(args):
    from token_routing_expert_gb300 import native

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    native.load()
    spec = W.WORKLOADS[args.config]
    if args.tokens > 0:
        spec = spec.with_(T=args.tokens)
    if args.experts > 0:
        spec = spec.with_(num_experts=args.experts)
    if args.capacity_factor > 0:
        spec = spec.with_(capacity_factor=args.capacity_factor)
    if args.fp8:
        spec = spec.with_(expert_fp8=native.EXPERT_FP8_ROWWISE)
    if args.mxfp8:
        spec = spec.with_(expert_fp8=native.EXPERT_MXFP8)
    if args.backward and args.mxfp8:
        raise SystemExit("--backward times the training path, which keeps bf16 pre-activations: not with --mxfp8")
    # each rank draws its own batch of tokens (weak scaling); weights are shared replicas
    inp = rank_inputs(spec, rank)
    cfg = native.config_from_spec(spec)
    wts = native.DeviceWeights.from_inputs(inp)
    if spec.expert_fp8 == native.EXPERT_MXFP8:
        wts.quantize_experts_mxfp8()   # pre-quantised expert weights, outside the timed region
    elif spec.expert_fp8:
        wts.quantize_experts_fp8()
    T = spec.T
    x = inp["x"].cuda()
    ws = native.workspace(cfg, T)
    out = torch.empty((T, spec.d_model), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    # working set: does it exceed L2?  (otherwise flush L2 between steps)
    L2 = torch.cuda.get_device_properties(local).L2_cache_size
    for _ in range(max(args.warmup, 1)):
        native.moe_layer_forward(cfg, wts, x, ws, out=out)
    torch.cuda.synchronize()
    if native.moe_get_status() != 0:
        raise SystemExit("device status error during warm-up")
    inter = native.layer_intermediates(cfg, T, ws)
    touched = int((inter["counts"] > 0).sum().item())
    alg_bytes = W.algorithmic_bytes(spec, touched)
    # rows the grouped GEMMs compute: each expert's rows rounded up to whole row tiles (256-row
    # CTA-pair tiles from 192 rows per expert on average, 128-row tiles below, as the library plans)
    counts_h = inter["counts"].long().cpu()
    rows_h = int(counts_h.sum().item())
    tile_rows = 256 if (rows_h >= 192 * spec.num_experts and spec.expert_fp8 != native.EXPERT_MXFP8) else 128
    padded_rows = int(((counts_h + tile_rows - 1) // tile_rows).sum().item()) * tile_rows
    flush = alg_bytes < 2 * L2
    flush_buf = torch.empty(2 * L2 // 4 + 1024, dtype=torch.float32, device="cuda") if flush else None

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(10)] for _ in range(args.steps)]
    for row in evs:  # create the underlying CUDA events
        for e in row:
            e.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local).start() if rank == 0 else None
    time.sleep(0.5 if clocks else 0)
    # the timed region: plain moe_layer_forward calls, nothing between the kernels of a step (its
    # kernels overlap their launches with the previous kernel's tail); with an L2 flush between
    # steps, events around each step leave the flush out
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] if flush else None
    t_wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        if flush:
            flush_buf.fill_(float(i))
            step_ev[i][0].record(stream)
        native.moe_layer_forward(cfg, wts, x, ws, out=out)
        if flush:
            step_ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    time.sleep(0.1 if clocks else 0)
    clock_info = clocks.stop(t_wall0, t_wall1) if clocks else None
    if native.moe_get_status() != 0:
        raise SystemExit("device status error in the timed region")
    ms = (sum(a.elapsed_time(b) for a, b in step_ev) / args.steps if flush
          else start.elapsed_time(end) / args.steps)

    # the per-stage split: the same steps again with events recorded at the stage boundaries
    for i in range(args.steps):
        if flush:
            flush_buf.fill_(float(i))
        native.moe_layer_forward_staged(cfg, wts, x, ws, evs[i], out=out)
    torch.cuda.synchronize()
    stage_ms = {}
    for s, name in enumerate(native.STAGES, start=1):
        stage_ms[name] = sum(evs[i][s - 1].elapsed_time(evs[i][s]) for i in range(args.steps)) / args.steps
    ms = max_over_ranks(ms, dist, "cuda")
    # the memory-bound stages against their own minimum bytes (inputs read once, outputs written once)
    Lr, R, E_ = spec.routed_dim, spec.rows, spec.num_experts
    stage_bytes = {
        "topk": T * E_ * 4 + T * spec.top_k * 8,                   # fp32 logits in; idx + weights out
        "permute": spec.T * spec.top_k * 4 + R * 8 + (2 * E_ + 1) * 4,   # idx in; gather, scatter, counts, offsets
        "combine": R * Lr * 2 + spec.T * spec.top_k * 8 + T * Lr * 2,  # Y rows, scatter + weights in; z out
    }
    stage_gbs = {k: v / (stage_ms[k] * 1e-3) / 1e9 for k, v in stage_bytes.items() if stage_ms[k] > 0}

    # end to end: pinned host input -> device, forward, output -> pinned host, every step
    x_host = inp["x"].pin_memory()
    # end to end through the host-batch entry point: every step copies its (T, d_model) input from
    # pinned host memory and its output back, overlapped with the neighbouring steps' compute
    x_hosts = [x_host, x_host.clone().pin_memory()]
    out_hosts = [torch.empty((T, spec.d_model), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    hws = native.host_workspace(cfg, T)
    native.moe_layer_forward_host_batches(cfg, wts, x_hosts, out_hosts, hws)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    native.moe_layer_forward_host_batches(cfg, wts, [x_hosts[i & 1] for i in range(args.steps)],
                                          [out_hosts[i & 1] for i in range(args.steps)], hws)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, "cuda")
    del hws
    if native.moe_get_status() != 0:
        raise SystemExit("device status error in the end-to-end region")

    bwd = None
    if args.backward:
        # backward of the combine and of the grouped SwiGLU experts on this batch (fresh dz each run)
        counts_d, offsets_d = inter["counts"], inter["offsets"]
        gather_d, scatter_d, w_d = inter["gather_idx"], inter["scatter_idx"], inter["weights"]
        y_d = inter["y"]
        xr_d = inter["x_routed"] if spec.latent_dim else x
        dz = torch.randn((T, spec.routed_dim), device="cuda").to(torch.bfloat16)
        dy_d = torch.empty_like(y_d)
        dw_d = torch.empty_like(w_d)
        bws = native.backward_workspace(cfg, T)
        # the training forward keeps the experts' pre-activations; timed against the plain forward
        preact = torch.empty((native.moe_permuted_rows(cfg, T), 2 * spec.hidden_size), dtype=torch.bfloat16,
                             device="cuda")
        fwd_out = torch.empty((T, spec.d_model), dtype=torch.bfloat16, device="cuda")

        logits_keep = torch.empty((T, spec.num_experts), dtype=torch.float32, device="cuda")

        def train_forward():
            native.moe_layer_forward_preact(cfg, wts, x, ws, out=fwd_out, preact=preact, logits=logits_keep)

        def plain_forward():
            native.moe_layer_forward(cfg, wts, x, ws, out=fwd_out)

        def timed(fn):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(args.steps):
                fn()
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / args.steps

        fwd_plain_ms, fwd_train_ms = timed(plain_forward), timed(train_forward)
        # the intermediates below are the last forward's (the same batch, so the same routing)
        dx_d = torch.empty((T, spec.routed_dim), dtype=torch.bfloat16, device="cuda")
        dwug = torch.empty((spec.num_experts, 2 * spec.hidden_size, spec.routed_dim), dtype=torch.float32, device="cuda")
        dwo = torch.empty((spec.num_experts, spec.routed_dim, spec.hidden_size), dtype=torch.float32, device="cuda")

        def backward_step():
            native.moe_combine_backward(cfg, dz, y_d, scatter_d, w_d, gather_idx=gather_d, dy=dy_d, dweights=dw_d)
            native.moe_grouped_swiglu_backward_preact(cfg, wts, xr_d, gather_d, offsets_d, scatter_d, dy_d, preact,
                                                      bws, dx_routed=dx_d, dw_up_gate=dwug, dw_out=dwo)

        def backward_step_recompute():
            native.moe_combine_backward(cfg, dz, y_d, scatter_d, w_d, gather_idx=gather_d, dy=dy_d, dweights=dw_d)
            native.moe_grouped_swiglu_backward(cfg, wts, xr_d, gather_d, offsets_d, scatter_d, dy_d, bws,
                                               dx_routed=dx_d, dw_up_gate=dwug, dw_out=dwo)

        bms = timed(backward_step)
        bms_re = timed(backward_step_recompute)
        del bws
        # the whole layer's backward (router and, when latent, the projections as well) after the
        # training forward above left its intermediates in ws
        train_forward()
        lbws = native.layer_backward_workspace(cfg, T)
        dout = torch.randn((T, spec.d_model), device="cuda").to(torch.bfloat16)
        ldx = torch.empty((T, spec.d_model), dtype=torch.bfloat16, device="cuda")

        def layer_backward_step():
            native.moe_layer_backward(cfg, wts, x, ws, preact, logits_keep, dout, lbws, dx=ldx)

        lms = timed(layer_backward_step)
        del lbws
        if native.moe_get_status() != 0:
            raise SystemExit("device status error in the backward")
        lflops = (12 * spec.rows * spec.routed_dim * spec.hidden_size + 4 * T * spec.num_experts * spec.d_model
                  + (8 * T * spec.d_model * spec.latent_dim if spec.latent_dim else 0))
        bflops = 12 * spec.rows * spec.routed_dim * spec.hidden_size
        bwd = {"ms": bms, "tflops": bflops / (bms * 1e-3) / 1e12, "algorithmic_flops": bflops,
               "ms_recompute": bms_re, "forward_ms": fwd_plain_ms, "forward_keep_preact_ms": fwd_train_ms,
               "layer_ms": lms, "layer_tflops": lflops / (lms * 1e-3) / 1e12, "layer_algorithmic_flops": lflops,
               "note": "combine backward + experts backward from the forward's kept pre-activations (dH, dX, "
                       "dW_out, dW_up_gate GEMMs = 12 R L h FLOPs); ms_recompute recomputes them instead "
                       "(4 R L h more); forward_keep_preact_ms is the layer forward that keeps them; layer_ms is "
                       "moe_layer_backward: the whole layer's backward (+ router and latent projections)"}

    # load-balancing counters on this batch's histogram (between-step work, timed on its own)
    counts = inter["counts"].clone()
    accum = torch.zeros(spec.num_experts, dtype=torch.int64, device="cuda")
    sbias = torch.zeros(spec.num_experts, dtype=torch.float32, device="cuda")
    imb = torch.empty(1, dtype=torch.float32, device="cuda")
    bal = {}
    # these kernels take microseconds: a captured graph keeps host launch cost out of the timing
    for name, fn in (("accumulate_counts_us", lambda: native.moe_accumulate_counts(counts, accum)),
                     ("load_imbalance_us", lambda: native.moe_load_imbalance(counts, out=imb)),
                     ("score_bias_update_us", lambda: native.moe_score_bias_update(accum, 1e-3, sbias))):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                fn()
        graph.replay()
        torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        graph.replay()
        b1.record(stream)
        torch.cuda.synchronize()
        bal[name] = 1e3 * b0.elapsed_time(b1) / args.steps
        del graph
    bal["load_imbalance"] = float(native.moe_load_imbalance(counts).item())
    bal["bound"] = f"launch latency ({spec.num_experts} counters)"

    peaks, peak_kind = read_peaks()
    decode = None
    if args.decode_config and args.decode_config != spec.name and args.tokens == 0 and args.experts == 0 and not (
            spec.expert_fp8 or spec.capacity_factor):
        decode = decode_pass(args, native, args.decode_config, peaks, dist)
    flops = W.algorithmic_flops(spec)
    dropped = 0
    if spec.capacity_factor > 0:
        cap = native.moe_expert_capacity(cfg, T)
        kept = int(torch.clamp(inter["counts"].long(), max=cap).sum().item())
        dropped = spec.rows - kept
        flops -= 6 * spec.routed_dim * spec.hidden_size * dropped   # dropped assignments do no expert work
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    gemm1_flops = 4 * spec.rows * spec.routed_dim * spec.hidden_size
    gemm1_ms = stage_ms["grouped_gemm1_swiglu"]
    achieved = gemm1_flops / (gemm1_ms * 1e-3) / 1e12
    # a timed region of seconds runs under the power cap: compare it with the sustained figure
    region_s = t_wall1 - t_wall0
    sustained = region_s > 0.25 and "bf16_tflops_sustained" in peaks
    peak_tf = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    peak_label = (f"{peak_kind} bf16 {'sustained' if sustained else 'burst'} (MEASURED_PEAKS.json; timed region "
                  f"{region_s:.2f} s)") if peak_kind == "measured" else "fallback 1.9 PFLOP/s bf16"
    gemm_peak, gemm_label = peak_tf, peak_label
    if spec.expert_fp8:
        # e4m3 tensor peak: the measured bf16 figure x the nominal e4m3 / bf16 ratio (4.5 / 2.25 PFLOP/s)
        gemm_peak, gemm_label = 2.0 * peak_tf, peak_label + " x 2 (nominal e4m3 / bf16 ratio)"
    # roofline of the layer: the slower of its FLOPs at the tensor peak and its bytes at HBM
    # bandwidth; with e4m3 experts their FLOPs run at the e4m3 peak and their weights are 1 byte
    expert_flops = 6 * spec.routed_dim * spec.hidden_size * spec.rows
    t_flops = flops / (peak_tf * 1e12)
    roof_bytes = alg_bytes
    if spec.expert_fp8:
        t_flops = (flops - expert_flops) / (peak_tf * 1e12) + expert_flops / (gemm_peak * 1e12)
        # e4m3 weights: 1 byte a value instead of 2 (MXFP8 adds a scale byte per 32 values)
        roof_bytes = alg_bytes - touched * 3 * spec.routed_dim * spec.hidden_size * (
            31 / 32 if spec.expert_fp8 == native.EXPERT_MXFP8 else 1)
    t_bytes = roof_bytes / (peaks["hbm_gbs"] * 1e9)
    bound_layer = "hbm" if t_bytes > t_flops else "tensor"
    roof_ms = 1e3 * max(t_bytes, t_flops)

    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": job_tokens_per_s(world, T, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("bf16 (experts MXFP8: e4m3, E8M0 scale per 32 values)" if spec.expert_fp8 == native.EXPERT_MXFP8
                  else "bf16 (experts e4m3 rowwise)" if spec.expert_fp8 else "bf16"),
        "data": "synthetic (seeded numpy PCG64 normals rounded to bf16; random-init weights)",
        "config": dict(bench_config(spec, world),
                       l2=("flushed between steps (working set below 2x L2)" if flush else
                           f"no flush: algorithmic bytes per step {alg_bytes / 1e6:.0f} MB > L2 {L2 / 1e6:.0f} MB")),
        "layer": {"tflops": tflops, "frac_bf16_peak": tflops / peak_tf, "bf16_peak": peak_tf, "gbs": gbs,
                  "frac_hbm_peak": gbs / peaks["hbm_gbs"], "bound": bound_layer,
                  "roofline_ms": roof_ms, "frac_of_roofline": roof_ms / ms, "experts_touched": touched,
                  "algorithmic_flops": flops, "algorithmic_bytes": alg_bytes,
                  "dropped_assignments": dropped},
        "stages_ms": stage_ms,
        "stages_note": "a separate pass over the same steps with events at the stage boundaries (they break the "
                       "launch overlap between kernels, so the stages add up to a little more than ms_per_step)"
                       + ("; MXFP8 experts: quantising x_routed counts in 'gather', GEMM 1's epilogue quantises H"
                          if spec.expert_fp8 == native.EXPERT_MXFP8 else
                          "; e4m3 experts: quantising x_routed counts in 'gather', quantising H in 'grouped_gemm2'"
                          if spec.expert_fp8 else ""),
        "stages_gbs": {"values": stage_gbs, "bytes": stage_bytes,
                       "hbm_peak": peaks["hbm_gbs"], "note": "each stage's own minimum bytes"},
        "balance": bal,
        "backward": bwd,
        "decode": decode,
        "roofline": {"kernel": "grouped GEMM 1 (SwiGLU fused, tcgen05" + (
                     ", MXFP8 block-scaled operands)" if spec.expert_fp8 == native.EXPERT_MXFP8 else
                     ", e4m3 operands)" if spec.expert_fp8 else ")"),
                     "bound": "tensor", "achieved": achieved, "peak": gemm_peak, "unit": "TFLOP/s",
                     "frac": achieved / gemm_peak,
                     **({} if spec.capacity_factor else {
                         "rows": rows_h, "tile_rows": tile_rows, "padded_rows": padded_rows,
                         "padding_frac": 1.0 - rows_h / padded_rows if padded_rows else 0.0,
                         "achieved_on_padded_rows": achieved * padded_rows / rows_h if rows_h else 0.0}),
                     "traffic": (None if spec.expert_fp8 or spec.capacity_factor or args.tokens or args.experts
                                 else kernel_traffic(spec.name)),
                     "peak_source": gemm_label},
        "e2e": {"value": job_tokens_per_s(world, T, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": out_hosts[0].numel() * 2,
                "api": "moe_layer_forward_host_batches (copies overlapped with neighbouring steps)"},
        "gpu_launches": args.steps * native.moe_layer_forward_launches(cfg, T),
        "clocks": clock_info,
    }
    if world == 1 and not args.no_cpu_baseline:
        n = min(T, args.cpu_tokens)
        rate, reps, secs = oracle_sample_rate(spec, inp, n, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"first {n} of {T} tokens, full float64 layer, {reps} reps in "
                                          f"{secs:.1f} s (numpy BLAS on all host cores)"}
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="latent_prefill", choices=sorted(W.WORKLOADS))
    ap.add_argument("--decode-config", default="latent_decode",
                    help="decode-shaped workload timed in the same run ('' to skip)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens per step instead of the workload's own T (for small profiling captures)")
    ap.add_argument("--experts", type=int, default=0,
                    help="number of experts instead of the workload's own (for small profiling captures)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--capacity-factor", type=float, default=0.0,
                    help="> 0: capacity-limited experts (dropping); default dropless")
    ap.add_argument("--ref-tokens", type=int, default=256, help="at most this many oracle tokens per step (reference arm)")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="reference arm: per-step sample sized so the K timed steps take about this long")
    ap.add_argument("--cpu-tokens", type=int, default=512, help="oracle sample for the cpu_baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward", action="store_true", help="also time the combine + experts backward")
    ap.add_argument("--fp8", action="store_true", help="experts on rowwise e4m3 operands")
    ap.add_argument("--mxfp8", action="store_true", help="experts on MXFP8 operands (E8M0 block scales)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
