#!/usr/bin/env python
"""Throughput of the DeepSeekMoE layer pass (router GEMM + biased group-limited
top-K, permute, grouped SwiGLU experts on the tensor cores, shared expert,
combine, bias update) on B300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config v3]
  python bench.py --impl reference ...     (the CPU oracle, timed on host cores)
  python bench.py --pass train ...         (forward + backward + bias update per step)

One step = one pass of the whole path over one batch of T tokens plus the
bias update.  For N > 1 (launched with torch.distributed.run), every rank
runs a replica on its own T tokens; the per-expert loads are summed over the
ranks before the bias update (scaling "weak").  Prints one JSON line on rank 0.

The headline is the V3-shaped layer (T=8192).  At N=1 the same line also
carries "workloads": every other synthetic workload measured in the same run
(tiny; mid, 50 bias-feedback steps; decode at T=64/256/1024; the drifting
100-step run), each with tokens/s, ms/step and its roofline fraction
(--no-workloads skips them).
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (V3-shaped, bf16) and % of tensor-core / HBM roofline"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
# DRAM bytes (read + write) per routed expert of the two expert-GEMM launches,
# from ncu dram__bytes on the 16-expert V3-shaped profiling case (d=7168,
# I=2048, ~256 rows per expert), scaled by the experts a launch processes.
# Must be re-measured whenever those kernels change.
GEMM_TRAFFIC_PER_EXPERT = (1.042770688e9 + 16.624128e6 + 0.504207872e9 + 49.14816e6) / 16
# The timed region's length decides which measured tensor peak a fraction is
# taken against: a region shorter than this runs at burst clocks (the peak of
# a kernel timed alone); a longer one settles at the power-capped clock (the
# sustained peak).
SUSTAINED_AFTER_S = 1.0
KERNELS_PER_STEP = 12  # router GEMM, selection, 4 permute, 2+2 grouped GEMM, combine, bias update
# backward: combine 1; routed: dh GEMM, SwiGLU, dv GEMM, 2 weight-gradient GEMMs; shared:
# the same 5; router 3; input gradient 1 (the forward keeps the pre-activations)
KERNELS_PER_BACKWARD = 15
METRIC_TRAIN = "MoE-layer forward+backward tokens/s (V3-shaped, bf16, all gradients)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="v3",
                    help="tiny | mid | v3 | v3_drift | v3_decode:<T>")
    ap.add_argument("--cpu-sample", type=int, default=8,
                    help="tokens the CPU oracle baseline processes (rank 0, N=1)")
    ap.add_argument("--ref-sample", type=int, default=2,
                    help="tokens per step for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--feedback-steps", type=int, default=None,
                    help="steps of the mid / drift feedback runs (default: the workload's)")
    ap.add_argument("--shared-as-routed", action="store_true",
                    help="serving layout: shared experts routed as experts E.. inside the grouped GEMM")
    ap.add_argument("--redundant", type=int, default=0,
                    help="serving layout: redundant expert copies, planned from warm-up loads")
    ap.add_argument("--shared-stream", action="store_true",
                    help="run the shared expert on a second stream")
    ap.add_argument("--precision", choices=["bf16", "fp8"], default="bf16",
                    help="expert GEMM inputs: bf16, or E4M3 with 1x128 / 128x128 scales")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "train"], default="forward",
                    help="train: each step is the forward pass, the backward pass (all "
                         "gradients) and the bias update")
    ap.add_argument("--standard-weights", action="store_true",
                    help="run the expert GEMMs on the [rows, cols] weight layout instead of the "
                         "box-contiguous copies (same results)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads measured next to the headline (N=1)")
    return ap.parse_args()


def load_config(name):
    from expert_ffn_layer_affinity_b300 import synth
    if name.startswith("v3_decode"):
        T = int(name.split(":")[1]) if ":" in name else 1024
        return synth.CONFIGS["v3_decode"].with_T(T)
    return synth.CONFIGS[name]


def router_extra(cfg):
    """1 when the router GEMM splits its reduction (a small kernel then adds
    the splits), else 0."""
    from expert_ffn_layer_affinity_b300 import _lib as L
    return 1 if L.moe_router_splits(cfg.T, cfg.d, cfg.E) > 1 else 0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"],
                    bf16_sust=p.get("bf16_tflops_sustained", p["bf16_tflops"]), src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sust=1400.0, src="fallback")


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count()


class ClockSampler:
    """nvidia-smi samples every 50 ms; stop() keeps those taken between
    mark_start() and mark_stop() (host wall clock)."""

    def __init__(self, index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.t0 = self.t1 = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu=timestamp,{CLOCK_FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "50",
                                       "-i", str(index)], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
            return
        deadline = time.time() + 5
        while time.time() < deadline and os.path.getsize(self.f.name) == 0:
            time.sleep(0.02)

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_stop(self):
        self.t1 = datetime.datetime.now()

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.1)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        mhz, mx, reasons, power = [], 0.0, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f")
                if self.t0 and self.t1 and not (self.t0 <= ts <= self.t1):
                    continue
                mhz.append(float(r[2]))
                mx = max(mx, float(r[3]))
                power.append(float(r[4]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz), "power_w_max": max(power) if power else None,
                "power_w_median": statistics.median(power) if power else None}


# --------------------------------------------------------------------------
def algorithmic(cfg, touched, fp8=False):
    """Per-call algorithmic work (bytes moved at least once, dense FLOPs).
    With fp8 the expert GEMMs read 1-byte weights and activations (scales
    are 1/128 or less of that and not counted) and the dispatch quantizes x
    (bf16 in, E4M3 out) before gathering 1-byte rows."""
    T, d, E, K, I, ns = cfg.T, cfg.d, cfg.E, cfg.K, cfg.I, cfg.n_shared
    R = T * K
    if fp8:
        return {
            "route": dict(flops=2.0 * T * d * E * 3,
                          bytes=T * d * 2 + 3 * E * d * 2 + 2 * T * E * 4 + T * K * 8),
            "permute": dict(flops=0.0, bytes=4 * R * 4 + T * d * 3 + T * d + R * d),
            "routed": dict(flops=6.0 * d * I * R,
                           bytes=3.0 * touched * I * d + R * d + R * I * (2 + 2 + 1 + 1) + R * d * 2),
            "shared": dict(flops=6.0 * d * I * ns * T,
                           bytes=3.0 * ns * I * d + T * d + T * ns * I * 6 + T * d * 2),
            "combine": dict(flops=0.0, bytes=(R + 2 * T) * d * 2 + T * K * 8),
        }
    return {
        "route": dict(flops=2.0 * T * d * E * 3,
                      bytes=T * d * 2 + 3 * E * d * 2 + 2 * T * E * 4 + T * K * 8),
        "permute": dict(flops=0.0, bytes=2 * R * 4 + T * d * 2 + R * d * 2 + 2 * R * 4),
        "routed": dict(flops=6.0 * d * I * R,
                       bytes=3.0 * touched * I * d * 2 + R * d * 2 + 2 * R * I * 2 + R * d * 2),
        "shared": dict(flops=6.0 * d * I * ns * T,
                       bytes=3.0 * ns * I * d * 2 + T * d * 2 + 2 * T * ns * I * 2 + T * d * 2),
        "combine": dict(flops=0.0, bytes=(R + 2 * T) * d * 2 + T * K * 8),
    }


def cpu_baseline(cfg, layer, x, n_tokens, fp8=False):
    """The oracle as it stands, timed on the host on `n_tokens` tokens of the
    first batch (expert weights are fetched to host memory, and for fp8
    quantized by the oracle, before timing)."""
    import numpy as np
    import torch
    from oracle import fp8_ref as f8
    from oracle import moe_ref as ref

    def f64(t):
        return ref.bf16_to_f64(t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16))

    rng = np.random.default_rng(0)
    tok = np.sort(rng.choice(x.shape[0], n_tokens, replace=False))
    x_h = x[torch.from_numpy(tok).to(x.device)].cpu()
    w_r = layer.w_r.cpu().numpy()
    bias = layer.bias.cpu().numpy()
    off = layer.logit_offset.cpu().numpy() if layer.logit_offset is not None else None
    # which experts the oracle will need: from its own routing (untimed pre-pass)
    s = ref.router_affinity64(f64(x_h), w_r, off)
    idx, _ = ref.select_experts(s, bias.astype(np.float64), cfg.K, cfg.n_groups, cfg.topk_groups,
                                cfg.route_scale, precision="fp64")
    host = {int(e): (layer.w1[e].cpu(), layer.w3[e].cpu(), layer.w2[e].cpu())
            for e in np.unique(idx)}
    shared_h = (layer.ws1.cpu(), layer.ws3.cpu(), layer.ws2.cpu())
    if fp8:
        hq = {e: f8.quantize_expert(*(f64(w) for w in ws)) for e, ws in host.items()}
        shq = f8.quantize_expert(*(f64(w) for w in shared_h))
    t0 = time.perf_counter()
    x64 = f64(x_h)
    s = ref.router_affinity64(x64, w_r, off)
    idx, gate = ref.select_experts(s, bias.astype(np.float64), cfg.K, cfg.n_groups,
                                   cfg.topk_groups, cfg.route_scale, precision="fp64")
    load = ref.expert_load(idx, cfg.E)
    ref.bias_update(load, bias, n_tokens, cfg.K, cfg.E, cfg.gamma)
    if fp8:
        f8.moe_output64_fp8(x64, idx, gate, lambda e: hq[e], shq, cfg.n_shared)
    else:
        ref.moe_output64(x64, idx, gate, lambda e: tuple(f64(w) for w in host[e]),
                         tuple(f64(w) for w in shared_h), cfg.n_shared)
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n_tokens} random tokens of the first {cfg.T}-token batch, full layer "
                      f"(routing, {cfg.K} routed + {cfg.n_shared} shared SwiGLU experts in fp64"
                      f"{' on E4M3-quantized operands' if fp8 else ''}, "
                      f"load count, bias update); {dt:.1f} s"}


def tensor_peak(pk, timed_s, fp8=False):
    """(peak TFLOP/s, description) for a tensor-bound fraction: the burst
    figure when the timed region is shorter than SUSTAINED_AFTER_S (clocks
    still at burst), else the sustained one; E4M3 counts 2 x bf16 (the
    nominal dense ratio, 4.5 / 2.25 PFLOP/s)."""
    burst = timed_s < SUSTAINED_AFTER_S
    peak = (pk["bf16"] if burst else pk["bf16_sust"]) * (2.0 if fp8 else 1.0)
    kind = (f"{'E4M3 = 2 x ' if fp8 else ''}bf16 {'burst' if burst else 'sustained'}, {pk['src']} "
            f"(timed region {timed_s:.3f} s {'<' if burst else '>='} {SUSTAINED_AFTER_S} s)")
    return peak, kind


def timed_steps(layer, cfg, xs, steps, warmup, names, group=None, local=0, redundant=0):
    """W warm-up steps, then `steps` timed steps of the whole path (route ->
    permute -> routed and shared experts -> combine -> bias update), each on
    the next batch of `xs`, bracketed by a barrier and a synchronize; per-call
    CUDA events on the launching stream.  The timed trajectory starts from the
    layer's initial bias."""
    import torch
    import torch.distributed as dist
    stream = torch.cuda.current_stream()
    bias0 = layer.bias.clone()

    def barrier():
        if group is not None:
            dist.barrier(device_ids=[local])

    for i in range(warmup):
        layer.step(xs[i % len(xs)], group=group)
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise RuntimeError(f"device status {layer.device_status()} during warm-up")
    if redundant:
        layer.plan_replicas(layer.load.cpu())    # copies placed from the warm-up loads
    touched = int((layer.load > 0).sum().item())
    layer.bias.copy_(bias0)
    stats_hist = torch.zeros(steps, 4, dtype=torch.float32, device="cuda")
    marks = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for n in names} for _ in range(steps)]
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    ev0.record(stream)
    for i in range(steps):
        layer.step(xs[i % len(xs)], group=group, marks=marks[i], stats_out=stats_hist[i])
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_stop()
    barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    if group is not None:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    per = {n: statistics.mean(m[n][0].elapsed_time(m[n][1]) for m in marks) for n in names}
    return dict(ms=ms, per=per, stats=stats_hist.cpu().numpy(), clocks=clk, touched=touched,
                status=layer.device_status())


def graphed_steps(layer, xs, steps, bias0):
    """The trajectory timed_steps times, from the same initial bias, with each
    step replayed from a CUDA graph captured beforehand for its batch (one
    host call per step instead of one per kernel).  Returns the time of the
    `steps` replays and their per-step load statistics."""
    import torch
    stats_hist = torch.zeros(steps, 4, dtype=torch.float32, device="cuda")
    graphs = [layer.capture_step(xs[i % len(xs)], stats_out=stats_hist[i]) for i in range(steps)]
    for _ in range(3):                       # warm-up replays, then back to the initial bias
        graphs[0].replay()
    layer.bias.copy_(bias0)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(0)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    ev0.record(stream)
    for g in graphs:
        g.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_stop()
    return dict(ms=ev0.elapsed_time(ev1), stats=stats_hist.cpu().numpy(), clocks=clocks.stop(),
                status=layer.device_status())


def workload_name(cfg):
    return (f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E} K={cfg.K} shared={cfg.n_shared} I={cfg.I} "
            f"groups={cfg.n_groups}/{cfg.topk_groups} scale={cfg.route_scale}")


def feedback_summary(cfg, stats):
    return {"steps": int(stats.shape[0]), "gamma": cfg.gamma,
            "max_over_mean_per_step": [round(float(v), 4) for v in stats[:, 2]],
            "cv_per_step": [round(float(v), 4) for v in stats[:, 3]],
            "first": round(float(stats[0, 2]), 4), "last": round(float(stats[-1, 2]), 4),
            "min": round(float(stats[:, 2].min()), 4), "max": round(float(stats[:, 2].max()), 4)}


def roofline_entry(cfg, res, steps, pk, fp8=False):
    """The dominant call's roofline: expert-weight streaming against HBM for
    the decode sizes, the routed expert GEMMs against the tensor peak
    otherwise, and none for the tiny layer (a launch-latency-bound pass of
    microseconds, where a fraction means nothing)."""
    per = res["per"]
    touched = res["touched"]
    timed_s = res["ms"] / 1e3
    if cfg.name == "tiny":
        return {"bound": "launch", "achieved": None, "peak": None, "unit": None, "frac": None,
                "traffic": None, "note": "launch-latency-bound microsecond pass: no roofline "
                                         "fraction is meaningful at this size"}
    if cfg.name == "v3_decode":
        # decode: the expert GEMMs stream the weights of the touched experts
        wbytes = 3.0 * (touched + cfg.n_shared) * cfg.I * cfg.d * (1 if fp8 else 2)
        gbs = wbytes / ((per["routed"] + per.get("shared", 0.0)) * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(gbs / pk["hbm"], 4), "traffic": None,
                "kernel": "moe_grouped_swiglu routed + shared (expert-weight streaming)",
                "peak_kind": f"HBM copy, {pk['src']}", "weight_bytes_per_step": wbytes}
    alg = algorithmic(cfg, touched, fp8)
    routed_tf = alg["routed"]["flops"] / (per["routed"] * 1e-3) / 1e12
    peak, kind = tensor_peak(pk, timed_s, fp8)
    tc_burst, tc_sust = (tensor_peak(pk, 0.0, fp8)[0], tensor_peak(pk, 1e9, fp8)[0])
    return {"bound": "tensor", "achieved": round(routed_tf, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(routed_tf / peak, 4),
            "traffic": (GEMM_TRAFFIC_PER_EXPERT * touched
                        if cfg.d == 7168 and cfg.I == 2048 and not fp8 else None),
            "kernel": ("moe_grouped_swiglu_fp8 (routed experts: GEMM1+SwiGLU, h quantization, "
                       "GEMM2 launches)" if fp8 else
                       "moe_grouped_swiglu (routed experts: GEMM1+SwiGLU and GEMM2 launches)"),
            "peak_kind": kind, "frac_of_burst": round(routed_tf / tc_burst, 4),
            "frac_of_sustained": round(routed_tf / tc_sust, 4)}


def layer_fraction(cfg, ms_step, timed_s, pk, fp8=False):
    """Whole-layer tensor fraction: the routed + shared expert FLOPs of a step
    over the step time."""
    tf = cfg.expert_flops() / (ms_step * 1e-3) / 1e12
    peak, kind = tensor_peak(pk, timed_s, fp8)
    return {"expert_tflops": round(tf, 1), "frac": round(tf / peak, 4), "peak": peak,
            "peak_kind": kind, "frac_of_burst": round(tf / tensor_peak(pk, 0.0, fp8)[0], 4),
            "frac_of_sustained": round(tf / tensor_peak(pk, 1e9, fp8)[0], 4)}


def kernel_table(cfg, res, fp8=False):
    alg = algorithmic(cfg, res["touched"], fp8)
    kernels = {}
    for n, ms in res["per"].items():
        a = alg[n]
        k = {"ms": round(ms, 4)}
        if ms > 0:
            if a["flops"]:
                k["tflops"] = round(a["flops"] / (ms * 1e-3) / 1e12, 2)
            k["gbs"] = round(a["bytes"] / (ms * 1e-3) / 1e9, 1)
        kernels[n] = k
    return kernels


def run_workloads(args, v3_layer, pk):
    """The other synthetic workloads, measured in the same run as the
    headline (N=1): tiny, mid (its 50 bias-feedback steps), decode at
    T = 64 / 256 / 1024 and the drifting 100-step run (both on the V3
    layer's weights, as the workloads define them)."""
    import torch
    from expert_ffn_layer_affinity_b300 import synth
    from expert_ffn_layer_affinity_b300.layer import MoELayer
    names = ["route", "permute", "routed", "shared", "combine"]
    out = {}

    def one(cfg, layer, xs, steps, warmup, graphs=False):
        bias0 = layer.bias.clone()
        res = timed_steps(layer, cfg, xs, steps, warmup, names)
        ms_step = res["ms"] / steps
        entry = {"workload": workload_name(cfg), "steps": steps, "warmup": warmup,
                 "value": round(cfg.T * steps / (res["ms"] / 1e3), 1), "unit": "tokens/s",
                 "ms_per_step": round(ms_step, 4),
                 "roofline": roofline_entry(cfg, res, steps, pk),
                 "kernels": kernel_table(cfg, res), "experts_touched": res["touched"],
                 "gpu_launches": (KERNELS_PER_STEP + router_extra(cfg)) * steps,
                 "device_status": res["status"], "clocks": res["clocks"]}
        if cfg.name not in ("tiny", "v3_decode"):
            entry["layer_tensor_frac"] = layer_fraction(cfg, ms_step, res["ms"] / 1e3, pk)
        if cfg.steps > 1:
            entry["feedback"] = feedback_summary(cfg, res["stats"])
        if graphs:
            # the same steps replayed from CUDA graphs: launch-bound steps lose
            # the host's per-call cost; the trajectory must match bit for bit
            g = graphed_steps(layer, xs, steps, bias0)
            entry["graphs"] = {
                "value": round(cfg.T * steps / (g["ms"] / 1e3), 1), "unit": "tokens/s",
                "ms_per_step": round(g["ms"] / steps, 4),
                "same_trajectory": bool((g["stats"] == res["stats"]).all()),
                "gpu_launches": (KERNELS_PER_STEP + router_extra(cfg)) * steps,
                "device_status": g["status"], "clocks": g["clocks"]}
        return entry

    for name in ("tiny", "mid"):
        cfg = synth.CONFIGS[name]
        p = synth.make_params(cfg, "cuda")
        layer = MoELayer(cfg, p)
        del p
        n_batches = cfg.steps if cfg.steps > 1 else 2
        xs = [synth.make_tokens(cfg, step=i, device="cuda") for i in range(n_batches)]
        out[name] = one(cfg, layer, xs, cfg.steps if cfg.steps > 1 else 50, 5, graphs=True)
        del layer, xs
        torch.cuda.empty_cache()
    # decode sizes and the drifting run share the V3 layer's weights
    v3_cfg, bias0 = v3_layer.cfg, v3_layer.bias.clone()
    for T in synth.DECODE_T:
        cfg = synth.CONFIGS["v3_decode"].with_T(T)
        v3_layer.cfg = cfg
        v3_layer.bias.copy_(bias0)
        xs = [synth.make_tokens(cfg, step=i, device="cuda", seed=100 + T) for i in range(2)]
        out[f"v3_decode:{T}"] = one(cfg, v3_layer, xs, 20, 5)
    cfg = synth.CONFIGS["v3_drift"]
    v3_layer.cfg = cfg
    v3_layer.bias.copy_(bias0)
    xs = [synth.make_tokens(cfg, step=i, device="cuda") for i in range(cfg.steps)]
    out["v3_drift"] = one(cfg, v3_layer, xs, cfg.steps, 3)
    del xs
    v3_layer.cfg = v3_cfg
    v3_layer.bias.copy_(bias0)
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist
    from expert_ffn_layer_affinity_b300 import synth
    from expert_ffn_layer_affinity_b300.layer import MoELayer

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    group = None
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        group = dist.group.WORLD
    cfg = load_config(args.config)
    p = synth.make_params(cfg, "cuda")            # identical replicas on every rank
    fp8 = args.precision == "fp8"
    layer = MoELayer(cfg, p, device=f"cuda:{local}", shared_stream=args.shared_stream,
                     shared_as_routed=args.shared_as_routed, n_redundant=args.redundant,
                     precision=args.precision,
                     tiled_weights=False if args.standard_weights else None)
    del p
    feedback = cfg.steps > 1                     # mid / drift: a bias-feedback run
    if feedback:
        # one fresh batch per step, all resident in HBM before timing
        args.steps = cfg.steps if args.feedback_steps is None else args.feedback_steps
        n_batches = args.steps
    else:
        n_batches = 2
    xs = [synth.make_tokens(cfg, step=i, device="cuda", seed=cfg.seed + 7777 * rank)
          for i in range(n_batches)]
    stream = torch.cuda.current_stream()
    names = ["route", "permute", "routed", "combine"]
    if not args.shared_as_routed:
        names.insert(3, "shared")

    def barrier():
        if group is not None:
            dist.barrier(device_ids=[local])

    res = timed_steps(layer, cfg, xs, args.steps, args.warmup, names, group=group, local=local,
                      redundant=args.redundant)
    ms = res["ms"]
    ms_step = ms / args.steps
    value = cfg.T * world * args.steps / (ms / 1e3)

    # end to end through the public API (HostPipeline): every step copies its
    # tokens from pinned host memory to the device and its output back, the
    # copies of neighbouring steps overlapping this step's compute
    e2e = None
    if not args.no_e2e and not feedback:
        from expert_ffn_layer_affinity_b300.layer import HostPipeline
        x_host = [x.cpu().pin_memory() for x in xs]
        out_host = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory()
                    for _ in range(2)]
        pipe = HostPipeline(layer, cfg.T)
        for i in range(3):
            pipe.step(i, x_host[i % n_batches], out_host[i % 2], group=group)
        pipe.finish()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            pipe.step(i, x_host[i % n_batches], out_host[i % 2], group=group)
        pipe.finish()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = e0.elapsed_time(e1)
        if group is not None:
            t = torch.tensor([ems], device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ems = float(t.item())
        nbytes = cfg.T * cfg.d * 2
        e2e = {"value": cfg.T * world * args.steps / (ems / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
               "ms_per_step": ems / args.steps,
               "api": "HostPipeline (pinned host buffers; copies overlap neighbouring steps)"}

    if rank != 0:
        if group is not None:
            dist.destroy_process_group()
        return
    pk = peaks()
    if "shared" not in res["per"]:
        res["per"]["shared"] = 0.0                # inside the routed call in the serving layout
    kernels = kernel_table(cfg, res, fp8)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 expert GEMMs (fp32 promotion), bf16 activations" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02) weights, random-init)",
        "config": {"workload": workload_name(cfg),
                   "tokens_per_rank": cfg.T, "parallelism": f"dp{world} (replicas, load all-reduce)",
                   "l2": "inputs larger than L2: 22.6 GB of expert weights streamed per step"
                   if cfg.d == 7168 else "two alternating token batches",
                   "shared_stream": bool(args.shared_stream),
                   "shared_as_routed": bool(args.shared_as_routed),
                   "redundant_experts": args.redundant,
                   "precision": args.precision,
                   "expert_weight_layout": "box-contiguous" if layer.tiled else "rows"},
        "roofline": roofline_entry(cfg, res, args.steps, pk, fp8),
        "layer_tensor_frac": layer_fraction(cfg, ms_step, ms / 1e3, pk, fp8),
        "kernels": kernels,
        "experts_touched": res["touched"],
        "hbm_kernels": {n: {"gbs": kernels[n]["gbs"],
                            "frac": round(kernels[n]["gbs"] / pk["hbm"], 4)}
                        for n in ("route", "permute", "combine")},
        "gpu_launches": (KERNELS_PER_STEP + router_extra(cfg) + 3 * fp8
                         - (3 if fp8 else 2) * bool(args.shared_as_routed)
                         + bool(args.redundant)) * args.steps,
        "device_status": res["status"],
        "clocks": res["clocks"],
        "e2e": e2e,
    }
    if feedback:
        line["feedback"] = feedback_summary(cfg, res["stats"])
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(cfg, layer, xs[0], args.cpu_sample, fp8)
    if (world == 1 and not args.no_workloads and args.config == "v3" and not fp8
            and not args.shared_as_routed and not args.redundant and not args.shared_stream):
        del xs
        line["workloads"] = run_workloads(args, layer, pk)
    print(json.dumps(line), flush=True)
    if group is not None:
        dist.destroy_process_group()


# --------------------------------------------------------------------------
def backward_bytes(cfg):
    """Algorithmic bytes of the routed weight-gradient GEMMs: fp32 gradients
    of every expert written once (zeros for an expert without tokens), and
    their bf16 operands read once."""
    T, d, E, K, I = cfg.T, cfg.d, cfg.E, cfg.K, cfg.I
    R = T * K
    return 4.0 * E * 3 * I * d + 2.0 * R * (d + I) + 2.0 * R * (2 * I + d)


def cpu_baseline_train(cfg, layer, x, dy, n_tokens):
    """The forward and backward oracles as they stand, on `n_tokens` tokens of
    the first batch (weights fetched to host memory before timing)."""
    import numpy as np
    import torch
    from oracle import moe_bwd_ref as B
    from oracle import moe_ref as ref

    def f64(t):
        return ref.bf16_to_f64(t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16))

    rng = np.random.default_rng(0)
    tok = torch.from_numpy(np.sort(rng.choice(x.shape[0], n_tokens, replace=False))).to(x.device)
    x_h, dy_h = x[tok].cpu(), dy[tok].cpu()
    w_r = layer.w_r.cpu().numpy()
    bias = layer.bias.cpu().numpy()
    off = layer.logit_offset.cpu().numpy() if layer.logit_offset is not None else None
    s = ref.router_affinity64(f64(x_h), w_r, off)
    idx, _ = ref.select_experts(s, bias.astype(np.float64), cfg.K, cfg.n_groups, cfg.topk_groups,
                                cfg.route_scale, precision="fp64")
    host = {int(e): (layer.w1[e].cpu(), layer.w3[e].cpu(), layer.w2[e].cpu())
            for e in np.unique(idx)}
    shared_h = (layer.ws1.cpu(), layer.ws3.cpu(), layer.ws2.cpu())
    t0 = time.perf_counter()
    x64, dy64 = f64(x_h), f64(dy_h)
    s = ref.router_affinity64(x64, w_r, off)
    idx, gate = ref.select_experts(s, bias.astype(np.float64), cfg.K, cfg.n_groups,
                                   cfg.topk_groups, cfg.route_scale, precision="fp64")
    experts = lambda e: tuple(f64(w) for w in host[e])
    shared = tuple(f64(w) for w in shared_h)
    ref.moe_output64(x64, idx, gate, experts, shared, cfg.n_shared)
    B.moe_layer_bwd64(x64, w_r, off, idx, cfg.route_scale, experts, shared, cfg.n_shared, dy64)
    ref.bias_update(ref.expert_load(idx, cfg.E), bias, n_tokens, cfg.K, cfg.E, cfg.gamma)
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n_tokens} random tokens of the first {cfg.T}-token batch: routing, "
                      f"forward and backward of the {cfg.K} routed + {cfg.n_shared} shared "
                      f"SwiGLU experts and the router in fp64, bias update; {dt:.1f} s"}


def run_train(args):
    """Forward + backward (+ bias update) per step, one GPU."""
    import torch
    from expert_ffn_layer_affinity_b300 import synth
    from expert_ffn_layer_affinity_b300.layer import MoELayer

    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and int(os.environ.get("RANK", "0")) != 0:
        return                                    # one replica measures (no cross-rank gradients)
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    cfg = load_config(args.config)
    p = synth.make_params(cfg, "cuda")
    layer = MoELayer(cfg, p, training=True)
    del p
    xs = [synth.make_tokens(cfg, step=i, device="cuda") for i in range(2)]
    dys = [synth.make_output_grad(cfg, step=i, device="cuda") for i in range(2)]
    stream = torch.cuda.current_stream()
    fnames = ["route", "permute", "routed", "shared", "combine"]
    bnames = ["bwd_combine", "bwd_routed_dgrad", "bwd_routed_wgrad", "bwd_shared", "bwd_router",
              "bwd_dx"]

    def step(i, marks=None):
        layer.forward(xs[i % 2], marks=marks)
        layer.backward(xs[i % 2], dys[i % 2], marks=marks)
        layer.bias_update(cfg.T)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise RuntimeError(f"device status {layer.device_status()} during warm-up")
    marks = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for n in fnames + bnames} for _ in range(args.steps)]
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    ev0.record(stream)
    for i in range(args.steps):
        step(i, marks[i])
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_stop()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    status = layer.device_status()
    per = {n: statistics.mean(m[n][0].elapsed_time(m[n][1]) for m in marks)
           for n in fnames + bnames}
    ms_step = ms / args.steps

    # end to end through the public API (HostPipeline, train=True): every step
    # copies x and dy from pinned host memory in and dx out, the copies of
    # neighbouring steps overlapping this step's compute
    e2e = None
    if not args.no_e2e:
        from expert_ffn_layer_affinity_b300.layer import HostPipeline
        x_host = [x.cpu().pin_memory() for x in xs]
        dy_host = [g.cpu().pin_memory() for g in dys]
        dx_host = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        pipe = HostPipeline(layer, cfg.T, train=True)
        for i in range(3):
            pipe.step(i, x_host[i % 2], dx_host[i % 2], dy_host=dy_host[i % 2])
        pipe.finish()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            pipe.step(i, x_host[i % 2], dx_host[i % 2], dy_host=dy_host[i % 2])
        pipe.finish()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = e0.elapsed_time(e1)
        nb = cfg.T * cfg.d * 2
        e2e = {"value": round(cfg.T * args.steps / (ems / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": 2 * nb, "d2h_bytes_per_step": nb,
               "ms_per_step": ems / args.steps,
               "api": "HostPipeline(train=True): x and dy copied in, dx copied out each step, "
                      "copies overlapping neighbouring steps (weight gradients stay on the device)"}

    pk = peaks()
    wg_bytes = backward_bytes(cfg)
    wg_gbs = wg_bytes / (per["bwd_routed_wgrad"] * 1e-3) / 1e9
    T, d, I, R = cfg.T, cfg.d, cfg.I, cfg.R
    dgrad_flops = 2.0 * R * d * I * 3           # dh; dv (2I deep)
    kernels = {n: {"ms": round(per[n], 4)} for n in fnames + bnames}
    kernels["bwd_routed_dgrad"]["tflops"] = round(dgrad_flops / (per["bwd_routed_dgrad"] * 1e-3)
                                                  / 1e12, 1)
    kernels["bwd_routed_wgrad"]["gbs"] = round(wg_gbs, 1)
    kernels["bwd_routed_wgrad"]["tflops"] = round(6.0 * R * d * I
                                                  / (per["bwd_routed_wgrad"] * 1e-3) / 1e12, 1)
    line = {
        "metric": METRIC_TRAIN, "value": round(cfg.T * args.steps / (ms / 1e3), 1),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (fp32 weight gradients)",
        "data": "synthetic (seeded N(0,1) tokens and output gradients, N(0,0.02) weights)",
        "config": {"workload": f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E} K={cfg.K} "
                               f"shared={cfg.n_shared} I={cfg.I} groups={cfg.n_groups}/"
                               f"{cfg.topk_groups} scale={cfg.route_scale}",
                   "pass": "train (forward, backward: dx, dW_r, dW1/dW3/dW2 of every routed "
                           "and shared expert; bias update)",
                   "l2": (f"inputs larger than L2 ({3 * cfg.E * cfg.I * cfg.d * 2 / 1e9:.1f} GB of "
                          f"expert weights read, {3 * cfg.E * cfg.I * cfg.d * 4 / 1e9:.1f} GB of fp32 "
                          f"weight gradients written per step)"
                          if 3 * cfg.E * cfg.I * cfg.d * 2 > 126e6 else
                          "two alternating batches (the workload fits in L2)")},
        "roofline": {"bound": "hbm", "achieved": round(wg_gbs, 1), "peak": pk["hbm"],
                     "unit": "GB/s", "frac": round(wg_gbs / pk["hbm"], 4), "traffic": None,
                     "kernel": "moe_grouped_gemm_wgrad, routed (dW2 and [dW1; dW3] launches)",
                     "peak_kind": f"HBM copy, {pk['src']}",
                     "bytes_per_launch_pair": wg_bytes},
        "kernels": kernels,
        "gpu_launches": (KERNELS_PER_STEP + router_extra(cfg) + KERNELS_PER_BACKWARD) * args.steps,
        "device_status": status,
        "clocks": clk,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_train(cfg, layer, xs[0], dys[0], args.cpu_sample)
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
def run_reference(args):
    """The CPU oracle on the host cores, one bounded sample of the workload per
    step: `ref_sample` tokens routed and run through their experts in fp64,
    then the load count and bias update."""
    import numpy as np
    import torch
    from expert_ffn_layer_affinity_b300 import synth
    from oracle import moe_ref as ref

    if int(os.environ.get("RANK", "0")) != 0:
        return
    cfg = load_config(args.config)
    n = args.ref_sample

    def f64(t):
        return ref.bf16_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))

    w_r, bias, off = synth.make_router(cfg, "cpu")
    w_r, bias = w_r.numpy(), bias.numpy()
    off = off.numpy() if off is not None else None
    shared = tuple(f64(w) for w in synth.make_shared(cfg, "cpu"))
    cache = {}

    def expert(e):
        if e not in cache:
            if len(cache) >= 48:
                cache.pop(next(iter(cache)))
            cache[e] = synth.make_expert(cfg, e, "cpu")
        return cache[e]

    times = []
    for step in range(args.warmup + args.steps):
        x = synth.make_tokens(cfg, step, "cpu", T=n)
        s = ref.router_affinity64(f64(x), w_r, off)
        pre_idx, _ = ref.select_experts(s, bias.astype(np.float64), cfg.K, cfg.n_groups,
                                        cfg.topk_groups, cfg.route_scale, precision="fp64")
        for e in np.unique(pre_idx):
            expert(int(e))                      # input generation, untimed
        t0 = time.perf_counter()
        x64 = f64(x)
        s = ref.router_affinity64(x64, w_r, off)
        idx, gate = ref.select_experts(s, bias.astype(np.float64), cfg.K, cfg.n_groups,
                                       cfg.topk_groups, cfg.route_scale, precision="fp64")
        ref.moe_output64(x64, idx, gate, lambda e: tuple(f64(w) for w in expert(e)), shared,
                         cfg.n_shared)
        load = ref.expert_load(idx, cfg.E)
        bias = ref.bias_update(load, bias, n, cfg.K, cfg.E, cfg.gamma)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = n * len(times) / total
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(times), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, random-init)",
        "config": {"workload": f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E} K={cfg.K} "
                               f"shared={cfg.n_shared} I={cfg.I} groups={cfg.n_groups}/"
                               f"{cfg.topk_groups} scale={cfg.route_scale}",
                   "sample_tokens_per_step": n},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{n} tokens per step of the {cfg.T}-token workload, "
                                   f"full layer in fp64 on the host"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.pass_ == "train":
        run_train(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
