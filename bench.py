#!/usr/bin/env python3
"""Benchmark of the sparse MoE FFN layer on GB300 (one JSON line on rank 0).

A step is one forward of the whole layer (router -> select -> group ->
experts -> combine, plus the shared expert) over one batch of synthetic
tokens already resident in HBM.  Steps rotate over several layers with
distinct weight memory (as consecutive MoE layers of a model would), so the
selected experts' weights of a step were not touched in the previous steps
and come from HBM, not L2.

Default workload: qwen35moe-shaped layer (H=2048, E=256, top-8, F=512,
shared expert 512, bf16 weights/activations, fp32 accumulation), decode
batch of 8 tokens; the 1- and 4-token batches are reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference]

--impl reference times the CPU oracle (the plain double-precision C
implementation) on the host cores on the same workload: the baseline the
GPU path is compared with.  Under torchrun (N > 1) every rank runs an
independent replica (tokens are independent, there is no exchange step);
value = tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE layer tokens/s"
UNIT = "tokens/s"

# workload -> (spec, timed tokens per step, extra token counts reported, layers rotated)
WORKLOADS = {
    "qwen_decode": (synth.QWEN, 8, (1, 4), 8),
    "qwen_prefill_zipf": (synth.QWEN_ZIPF, 4096, (), 4),
    "gptoss_decode": (synth.GPTOSS, 1, (64,), 4),
    "gptoss_prefill": (synth.GPTOSS, 2048, (), 3),
    "mixtral_decode": (synth.MIXTRAL, 1, (16, 256), 3),
    "mixtral_prefill": (synth.MIXTRAL, 4096, (16384,), 2),
    "gptoss_mxfp4_decode": (synth.GPTOSS_MXFP4, 1, (4, 16), 6),
}
N_BATCHES = 16  # distinct token batches cycled through


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# distributed helpers (host-side only; gloo on CPU tensors)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws):
    if ws <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return dist


def reduce_max(value: float, dist=None) -> float:
    """Maximum of `value` over ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist=None):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks sampler
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------
def oracle_rate(spec, w, budget_s: float = 12.0, max_tokens: int = 1 << 16, seed: int = 1):
    """Tokens/s of the oracle (all host cores) on a sample of tokens drawn like
    the workload's, sized to take about budget_s seconds."""
    import oracle
    orc = oracle.Oracle(spec, w)
    cores = oracle.max_threads()
    n = max(1, cores)
    x = synth.make_x(spec, n, seed=seed)
    t0 = time.perf_counter()
    orc.forward(x)
    per_tok = (time.perf_counter() - t0) / n
    m = int(max(n, min(max_tokens, budget_s / max(per_tok, 1e-9))))
    x = synth.make_x(spec, m, seed=seed, first_token=n)
    t0 = time.perf_counter()
    orc.forward(x)
    dt = time.perf_counter() - t0
    return m / dt, cores, m, dt


def _spec_dtype(spec):
    if spec.expert_format == "mxfp4":
        return "mxfp4-f16"  # MXFP4 expert weights widened to f16 for the MMA, fp32 accumulation
    return "bf16" if spec.dtype == "bf16" else "f32"


def run_reference(args, spec, T):
    """--impl reference: the oracle timed per step on the host cores."""
    import oracle
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = synth.make_weights(spec, seed=0)
    x_pool = synth.make_x(spec, T * N_BATCHES, seed=0)
    orc = oracle.Oracle(spec, w)
    cores = oracle.max_threads()
    # per-token cost probe, then tokens per step so the whole run stays near a minute
    t0 = time.perf_counter()
    orc.forward(np.ascontiguousarray(x_pool[:min(T, cores)]))
    per_tok = (time.perf_counter() - t0) / min(T, cores)
    steps_total = args.steps + args.warmup
    tps = int(max(1, min(T, 60.0 / max(per_tok * steps_total, 1e-9))))
    for i in range(args.warmup):
        b = (i % N_BATCHES) * T
        orc.forward(np.ascontiguousarray(x_pool[b:b + tps]))
    t0 = time.perf_counter()
    for i in range(args.steps):
        b = (i % N_BATCHES) * T
        orc.forward(np.ascontiguousarray(x_pool[b:b + tps]))
    dt = time.perf_counter() - t0
    value = tps * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{spec.name}, {T} tokens per step", "tokens_per_step_timed": tps},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{tps} of the {T} tokens of each step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def _traffic_from_profiles(kernel: str, workload: str):
    """dram bytes per launch recorded under profiles/ for (kernel, workload),
    if the kernel source has not changed since (its sha256 is recorded)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 5 and cells[0] == kernel and cells[1] == workload:
            src, sha = cells[3], cells[4]
            p = os.path.join(ROOT, src)
            if not os.path.exists(p):
                return None
            if hashlib.sha256(open(p, "rb").read()).hexdigest()[:16] != sha:
                return None
            try:
                return float(cells[2])
            except ValueError:
                return None
    return None


def run_ours(args, spec, T, extra_T, n_layers, workload):
    import torch
    import sparse_mixture_experts_gb300 as moe
    from sparse_mixture_experts_gb300 import build as libbuild

    ws, rank, local = dist_env()
    dist = dist_init(ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not libbuild.up_to_date():
        if rank == 0:
            libbuild.build()
        barrier(dist)
    hbm_peak, tc_peak, tc_sustained, peak_src = _peaks()
    eb = 2 if spec.dtype == "bf16" else 4
    Tmax = max((T,) + tuple(extra_T))

    # ---- layers with distinct weight memory, token batches ----
    w = synth.make_weights(spec, seed=0)
    wt = {}
    for k, v in w.items():
        t = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16 else torch.from_numpy(v)
        wt[k] = t.to(dev)
    mxfp4 = spec.expert_format == "mxfp4"
    if mxfp4:  # the ABI takes the MXFP4 blocks in the gate_up_w / down_w slots
        wt["gate_up_w"] = wt.pop("gate_up_blocks")
        wt["down_w"] = wt.pop("down_blocks")
    cfg = moe.MoEConfig(
        hidden=spec.hidden, n_expert=spec.n_expert, top_k=spec.top_k, expert_ff=spec.expert_ff,
        shared_ff=spec.shared_ff,
        router_mode=moe.ROUTER_SOFTMAX_TOPK if spec.router_mode == "softmax_topk" else moe.ROUTER_TOPK_SOFTMAX,
        norm_topk_prob=spec.norm_topk_prob, weights_scale=spec.weights_scale,
        act=moe.ACT_SWIGLU if spec.act == "swiglu" else moe.ACT_CLAMP_GLU, act_alpha=spec.act_alpha,
        act_limit=spec.act_limit, has_bias=spec.has_bias, gate_up_interleaved=spec.gate_up_interleaved,
        w_dtype=moe.DT_MXFP4 if mxfp4 else (moe.DT_BF16 if spec.dtype == "bf16" else moe.DT_F32),
        act_dtype=moe.DT_BF16 if spec.dtype == "bf16" else moe.DT_F32, out_dtype=moe.DT_F32, max_tokens=Tmax)
    layers = [moe.MoELayer(cfg, wt, device=dev) for _ in range(n_layers)]
    del wt
    torch.cuda.empty_cache()
    x_np = synth.make_x(spec, Tmax * N_BATCHES, seed=1 + rank)
    xt = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16) if x_np.dtype == np.uint16 else \
        torch.from_numpy(x_np)
    x_dev = xt.to(dev)
    out = torch.empty((Tmax, spec.hidden), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i, n_tok):
        b = (i % N_BATCHES) * Tmax
        layers[i % n_layers].forward(x_dev[b:b + n_tok], out[:n_tok], stream)

    def timed(n_tok, K):
        barrier(dist)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K):
            step(i, n_tok)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1)
        barrier(dist)
        return reduce_max(ms, dist)

    # ---- warm-up, clock window, timed region ----
    for i in range(max(3, args.warmup)):
        step(i, T)
    torch.cuda.synchronize(dev)
    for l in layers:
        l.status()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    t_load0 = time.time()
    t_end = time.time() + 1.0
    i = 0
    while time.time() < t_end:           # bring the clocks to their loaded state
        step(i, T)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize(dev)
    ms_total = timed(T, args.steps)
    launches = layers[(args.steps - 1) % n_layers].last_launch_count
    t_end = time.time() + 0.3
    while time.time() < t_end:
        step(i, T)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    t_load1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_load0, t_load1)
    ms_per_step = ms_total / args.steps
    value = ws * T * args.steps / (ms_total / 1e3)

    # ---- realised routing: distinct experts per batch ----
    distinct = []
    rows_per_batch = []
    for bi in range(N_BATCHES):
        b = bi * Tmax
        layers[0].forward(x_dev[b:b + T], out[:T], stream)
        c = layers[0].expert_counts(stream).cpu().numpy()
        distinct.append(int((c > 0).sum()))
        rows_per_batch.append(int(c.sum()))
    batches_used = [i % N_BATCHES for i in range(args.steps)]
    d_avg = float(np.mean([distinct[b] for b in batches_used]))
    H, F, Fs, E = spec.hidden, spec.expert_ff, spec.shared_ff, spec.n_expert
    # weight bytes a step reads per selected expert (MXFP4: half a byte per code
    # and a scale byte per 32 codes; biases are fp32 in the layer)
    wel = (0.5 + 1.0 / 32) if mxfp4 else eb
    per_expert_up = 2 * F * H * wel + (2 * F * 4 if spec.has_bias else 0)
    per_expert_down = H * F * wel + (H * 4 if spec.has_bias else 0)
    router_bytes = (E + (1 if Fs else 0)) * H * eb
    shared_bytes = 3 * Fs * H * eb
    step_bytes = d_avg * (per_expert_up + per_expert_down) + router_bytes + shared_bytes + T * H * (eb + 4)
    flops_routed = 2.0 * T * spec.top_k * 3 * H * F
    step_flops = flops_routed + 2.0 * T * 3 * H * Fs + 2.0 * T * H * E

    # ---- per-kernel device time (separate pass with events, same steps) ----
    for l in layers:
        l.timing_enable(args.steps + 8)
    for j in range(args.steps):
        step(j, T)
    torch.cuda.synchronize(dev)
    ktimes = {}
    for l in layers:
        for k, (ms, n) in l.timing_read().items():
            a, b = ktimes.get(k, (0.0, 0))
            ktimes[k] = (a + ms, b + n)
        l.timing_enable(0)
    kernel_avg_us = {k: (1e3 * ms / n if n else None) for k, (ms, n) in ktimes.items()}
    total_k = sum(ms for ms, _ in ktimes.values())
    kernel_share = {k: (ms / total_k if total_k else None) for k, (ms, _) in ktimes.items()}
    top = max((k for k in ktimes if ktimes[k][1]), key=lambda k: ktimes[k][0])
    if ktimes.get("experts", (0, 0))[1] or ktimes.get("experts_mxfp4", (0, 0))[1]:
        path = "weight-streaming tensor-core"
    elif ktimes.get("fused", (0, 0))[1]:
        path = "fused"
    elif ktimes.get("gather", (0, 0))[1]:
        path = "tensor-core"
    else:
        path = "stream"
    decode_like = path != "tensor-core"
    up_rows = T * spec.top_k
    if top in ("fused", "experts", "experts_mxfp4"):
        # all expert weights of the step stream through this one kernel
        alg = step_bytes - (router_bytes if top != "fused" else 0)
        bound, unit, peak = "hbm", "GB/s", hbm_peak
        achieved = alg / (kernel_avg_us[top] * 1e-6) / 1e9
    elif top in ("up", "down"):
        # bytes and flops of this kernel; the larger of its two floors names the bound
        hrows = (up_rows + T) * max(F, Fs) * eb
        if top == "up":
            kbytes = d_avg * per_expert_up + 2 * Fs * H * eb + (T if decode_like else up_rows + T) * H * eb + hrows
            kflops = 2.0 * up_rows * 2 * F * H + 2.0 * T * 2 * Fs * H
        else:
            ys = (up_rows + T) * H * (4 if decode_like else eb)
            kbytes = d_avg * per_expert_down + Fs * H * eb + hrows + ys
            kflops = 2.0 * up_rows * F * H + 2.0 * T * Fs * H
        kt = kernel_avg_us[top] * 1e-6
        if kbytes / (hbm_peak * 1e9) >= kflops / (tc_peak * 1e12):
            alg, bound, unit, peak = kbytes, "hbm", "GB/s", hbm_peak
            achieved = alg / kt / 1e9
        else:
            alg, bound, unit, peak = kflops, "tensor", "TFLOP/s", tc_peak
            achieved = alg / kt / 1e12
    else:
        alg, bound, unit, peak, achieved = None, "hbm", "GB/s", hbm_peak, None
    traffic = _traffic_from_profiles(top, workload)
    roofline = {"kernel": top, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                "algorithmic_per_launch": alg, "peak_source": peak_src}
    step_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9
    step_tflops = step_flops / (ms_per_step * 1e-3) / 1e12
    t_hbm = step_bytes / (hbm_peak * 1e9)
    t_tc = step_flops / (tc_peak * 1e12)
    step_roofline = {"bytes": step_bytes, "flops": step_flops, "achieved_gbs": step_gbs,
                     "hbm_frac": step_gbs / hbm_peak, "achieved_tflops": step_tflops,
                     "tc_frac": step_tflops / tc_peak,
                     "frac_of_max_floor": max(t_hbm, t_tc) / (ms_per_step * 1e-3)}

    # ---- extra token counts of the same workload ----
    extra = {}
    for n_tok in extra_T:
        for j in range(max(3, args.warmup)):
            step(j, n_tok)
        ms = timed(n_tok, args.steps)
        d = []
        for bi in range(N_BATCHES):
            b = bi * Tmax
            layers[0].forward(x_dev[b:b + n_tok], out[:n_tok], stream)
            d.append(int((layers[0].expert_counts(stream).cpu().numpy() > 0).sum()))
        dd = float(np.mean([d[i % N_BATCHES] for i in range(args.steps)]))
        by = dd * (per_expert_up + per_expert_down) + router_bytes + shared_bytes + n_tok * H * (eb + 4)
        fl = 2.0 * n_tok * spec.top_k * 3 * H * F + 2.0 * n_tok * 3 * H * Fs + 2.0 * n_tok * H * E
        mps = ms / args.steps
        extra[str(n_tok)] = {"tokens_per_s": ws * n_tok / (mps * 1e-3), "ms_per_step": mps,
                             "distinct_experts": dd, "hbm_frac": by / (mps * 1e-3) / 1e9 / hbm_peak,
                             "tc_frac": fl / (mps * 1e-3) / 1e12 / tc_peak}

    # ---- end to end through the C ABI with host buffers ----
    x_host = xt[:Tmax * N_BATCHES].pin_memory()
    out_host = torch.empty((Tmax, spec.hidden), dtype=torch.float32).pin_memory()
    for j in range(max(3, args.warmup)):
        b = (j % N_BATCHES) * Tmax
        layers[j % n_layers].forward_host(x_host[b:b + T], out_host[:T], stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for j in range(args.steps):
        b = (j % N_BATCHES) * Tmax
        layers[j % n_layers].forward_host(x_host[b:b + T], out_host[:T], stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1), dist)
    for l in layers:
        l.status()

    # ---- CPU baseline (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, cores, m, dt = oracle_rate(spec, w, budget_s=args.cpu_budget)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{m} tokens drawn like this workload's, one oracle call over all cores ({dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": _spec_dtype(spec), "data": "synthetic",
            "config": {"workload": f"{spec.name}, {T} tokens per step", "tokens_per_step": T,
                       "layers_rotated": n_layers,
                       "l2": (f"inputs larger than L2: steps rotate over {n_layers} layers with distinct weight "
                              f"memory ({layers[0].device_bytes * n_layers / 1e9:.1f} GB)"),
                       "token_batches": N_BATCHES, "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "distinct_experts_per_step": d_avg, "path": path},
            "roofline": roofline,
            "step_roofline": step_roofline,
            "kernels": {k: {"avg_us": kernel_avg_us[k], "share": kernel_share[k], "launches": ktimes[k][1]}
                        for k in ktimes if ktimes[k][1]},
            "cpu_baseline": cpu,
            "e2e": {"value": ws * T * args.steps / (e2e_ms / 1e3), "unit": UNIT,
                    "h2d_bytes_per_step": T * spec.hidden * eb, "d2h_bytes_per_step": T * spec.hidden * 4},
            "gpu_launches": launches * args.steps,
            "clocks": clocks,
            "other_token_counts": extra,
        }
        print(json.dumps(line), flush=True)
    for l in layers:
        l.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="qwen_decode")
    ap.add_argument("--tokens", type=int, default=0, help="override the timed tokens per step")
    ap.add_argument("--layers", type=int, default=0, help="override the number of rotated layers")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    spec, T, extra, n_layers = WORKLOADS[args.workload]
    if args.tokens:
        T, extra = args.tokens, ()
    if args.layers:
        n_layers = args.layers
    if args.impl == "reference":
        return run_reference(args, spec, T)
    return run_ours(args, spec, T, extra, n_layers, args.workload)


if __name__ == "__main__":
    sys.exit(main())
