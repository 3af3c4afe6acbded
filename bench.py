#!/usr/bin/env python3
"""Benchmark of the sparse MoE FFN layer on GB300 (one JSON line on rank 0).

A step is one forward of the whole layer (router -> select -> group ->
experts -> combine, plus the shared expert) over one batch of synthetic
tokens already resident in HBM.  Steps rotate over several layers with
distinct weight memory (as consecutive MoE layers of a model would), so the
selected experts' weights of a step were not touched in the previous steps
and come from HBM, not L2.

Headline workload: qwen35moe-shaped layer (H=2048, E=256, top-8, F=512,
shared expert 512, bf16 weights/activations, fp32 accumulation), decode
batch of 8 tokens; the 1- and 4-token batches are reported beside it.

The same run then measures every layer configuration at its full sizes, one
layer set at a time (created, timed, freed), under "workloads": the tiny fp32
layer, the qwen35moe-shaped layer (decode, and Zipf-skewed prefill of 4096
tokens), the gpt-oss-20b-shaped layer (1, 64, 2048 tokens; also with MXFP4
experts), and the mixtral-shaped token sweep (1 .. 16384).  Each entry gives
the step time (mean of the bracketed steps and median of per-step events),
tokens/s, the step's fraction of its roofline floor max(t_HBM, t_TC), the
dominant kernel's roofline, per-kernel times, the clocks seen, the realised
expert load, and the oracle's single-core and all-core rates.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-workloads]

--gpus N without torchrun starts N replica processes (one per GPU) through
torch.distributed.run; under torchrun WORLD_SIZE must equal N.  Tokens are
independent and every replica holds all weights, so the replicas exchange
nothing on the data path: value = tokens of all ranks / the slowest rank's
time.  --impl reference times the CPU oracle (the plain double-precision C
implementation) on the host cores on the headline workload.
"""
from __future__ import annotations

import argparse
import json
import os
import socket
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
    "gptoss_mxfp4_prefill": (synth.GPTOSS_MXFP4, 2048, (64,), 3),
    "qwen_q4_decode": (synth.QWEN_Q4, 8, (1,), 8),
    "qwen_streamed_decode": (synth.QWEN_STREAMED, 8, (1,), 4),
    "gptoss_q4_prefill": (synth.GPTOSS_Q4, 2048, (16,), 3),
    "tiny": (synth.TINY, 16, (), 1),
}

# every layer configuration at its full sizes: name -> (spec, token counts, layers rotated)
SWEEP = {
    "tiny_f32": (synth.TINY, (16,), 1),
    "qwen35moe_decode": (synth.QWEN, (1, 4, 8), 8),
    "qwen35moe_prefill_zipf": (synth.QWEN_ZIPF, (4096,), 4),
    "gptoss20b": (synth.GPTOSS, (1, 64, 2048), 4),
    "gptoss20b_mxfp4": (synth.GPTOSS_MXFP4, (1, 4, 16, 64, 2048), 4),
    "qwen35moe_q4": (synth.QWEN_Q4, (1, 8, 300), 8),
    "qwen35moe_streamed": (synth.QWEN_STREAMED, (1, 8), 4),
    "gptoss20b_q4": (synth.GPTOSS_Q4, (1, 16, 2048), 4),
    "mixtral": (synth.MIXTRAL, (1, 16, 256, 4096, 16384), 2),
}
# the headline workload's sweep entry (measured once, reported in both places)
HEADLINE_SWEEP = {"qwen_decode": "qwen35moe_decode"}

N_BATCHES = 16  # distinct token batches cycled through
MEDIAN_MIN_STEPS = 50


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# process launch and distributed helpers (host-side only; gloo on CPU tensors)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launcher_cmd(n: int, argv, port: int | None = None):
    """The command that runs this script as n replica ranks on one node."""
    port = _free_port() if port is None else port
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]


def check_world(gpus: int, environ=None) -> str:
    """'spawn' when this process must start `gpus` replica ranks itself, 'run'
    when it is one of the ranks (or the only process).  Raises when torchrun
    started a different number of ranks than --gpus asks for."""
    env = os.environ if environ is None else environ
    if "WORLD_SIZE" not in env:
        return "spawn" if gpus > 1 else "run"
    ws = int(env["WORLD_SIZE"])
    if ws != gpus:
        raise SystemExit(f"bench.py: --gpus {gpus} but WORLD_SIZE={ws}; launch one rank per GPU")
    return "run"


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


def run_check_launch():
    """--check-launch: every rank joins the gloo group and rank 0 prints the
    world size and the sum of the ranks (no GPU work)."""
    import torch
    ws, rank, _ = dist_env()
    dist = dist_init(ws)
    t = torch.tensor([float(rank)], dtype=torch.float64)
    if dist is not None:
        dist.all_reduce(t)
    if rank == 0:
        print(json.dumps({"world_size": ws, "rank_sum": int(t.item())}), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


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
        for ts, line in list(self.lines):
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
def oracle_rate(spec, w, budget_s: float = 12.0, max_tokens: int = 1 << 16, seed: int = 1, n_threads: int = 0):
    """Tokens/s of the oracle on a sample of tokens drawn like the workload's,
    sized to take about budget_s seconds; n_threads 0 = all host cores."""
    import oracle
    orc = oracle.Oracle(spec, w)
    cores = oracle.max_threads() if n_threads <= 0 else n_threads
    n = max(1, cores)
    x = synth.make_x(spec, n, seed=seed)
    t0 = time.perf_counter()
    orc.forward(x, n_threads=cores)
    per_tok = (time.perf_counter() - t0) / n
    m = int(max(n, min(max_tokens, budget_s / max(per_tok, 1e-9))))
    x = synth.make_x(spec, m, seed=seed, first_token=n)
    t0 = time.perf_counter()
    orc.forward(x, n_threads=cores)
    dt = time.perf_counter() - t0
    return m / dt, cores, m, dt


def cpu_baselines(spec, w, budget_all: float, budget_one: float):
    """The oracle's all-core and single-core rates (a baseline, not a target)."""
    rate, cores, m, dt = oracle_rate(spec, w, budget_s=budget_all)
    out = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{m} tokens drawn like this workload's, one oracle call over all cores ({dt:.1f} s)"}
    if budget_one > 0:
        r1, _, m1, dt1 = oracle_rate(spec, w, budget_s=budget_one, n_threads=1)
        out["single_core"] = {"value": r1, "unit": UNIT, "cores": 1,
                              "sample": f"{m1} tokens on one host core ({dt1:.1f} s)"}
    return out


def _spec_dtype(spec):
    if spec.expert_format == "mxfp4":
        return "mxfp4-bf16"  # MXFP4 expert weights widened to bf16 on chip for the MMA, fp32 accumulation
    if spec.expert_format == "q4":
        return "q4-bf16"     # Q4 expert records widened (rounded) to bf16 on chip, fp32 accumulation
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
# roofline model: algorithmic bytes and flops per step and per kernel launch
# ---------------------------------------------------------------------------
def _traffic_from_profiles(kernel: str, workload: str, tokens: int):
    """dram bytes per launch recorded under profiles/ for (kernel, workload,
    tokens per step), if the kernel source has not changed since (its
    sha256[:16] is recorded)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 6 and cells[0] == kernel and cells[1] == workload and cells[2] == str(tokens):
            src, sha = cells[4], cells[5]
            p = os.path.join(ROOT, src)
            if not os.path.exists(p):
                return None
            if hashlib.sha256(open(p, "rb").read()).hexdigest()[:16] != sha:
                return None
            try:
                return float(cells[3])
            except ValueError:
                return None
    return None


class Model:
    """Algorithmic bytes and flops of one layer configuration.

    Weight bytes of a step count each selected expert once (the realised
    number of distinct experts), the router and the shared expert, plus the
    tokens in and the fp32 output.  Flops are the routed ones (2 T k 3 H F),
    the shared expert's and the router's: not a dense all-experts count."""

    def __init__(self, spec):
        self.spec = spec
        self.mx = spec.expert_format in ("mxfp4", "q4")
        self.eb = 2 if spec.dtype == "bf16" else 4
        H, F, Fs, E = spec.hidden, spec.expert_ff, spec.shared_ff, spec.n_expert
        # MXFP4: half a byte per code and a scale byte per 32; Q4: a two-byte scale per 32
        wel = {"mxfp4": 0.5 + 1.0 / 32, "q4": 0.5 + 2.0 / 32}.get(spec.expert_format, self.eb)
        self.up_per_expert = 2 * F * H * wel + (2 * F * 4 if spec.has_bias else 0)
        self.down_per_expert = H * F * wel + (H * 4 if spec.has_bias else 0)
        self.router = (E + (1 if Fs else 0)) * H * self.eb
        self.shared = 3 * Fs * H * self.eb

    def step_bytes(self, T, d):
        H = self.spec.hidden
        return d * (self.up_per_expert + self.down_per_expert) + self.router + self.shared + T * H * (self.eb + 4)

    def step_flops(self, T):
        s = self.spec
        return 2.0 * T * s.top_k * 3 * s.hidden * s.expert_ff + 2.0 * T * 3 * s.hidden * s.shared_ff + \
            2.0 * T * s.hidden * s.n_expert

    def kernel(self, kind, T, d):
        """(bytes, flops) one launch of kernel `kind` must move / compute."""
        s, eb = self.spec, self.eb
        H, F, Fs, K = s.hidden, s.expert_ff, s.shared_ff, s.top_k
        rows = T * K + (T if Fs else 0)              # routed rows + the shared expert's
        hbytes = rows * max(F, Fs) * 2               # h, bf16
        if kind in ("experts", "experts_mxfp4", "experts_q4"):  # decode: the whole layer after the router
            return self.step_bytes(T, d) - self.router, self.step_flops(T) - 2.0 * T * H * s.n_expert
        if kind == "fused":
            return self.step_bytes(T, d), self.step_flops(T)
        if kind == "up":
            b = d * self.up_per_expert + 2 * Fs * H * eb + rows * H * eb + hbytes
            return b, 2.0 * T * K * 2 * F * H + 2.0 * T * 2 * Fs * H
        if kind == "down":
            b = d * self.down_per_expert + Fs * H * eb + hbytes + (T * (K + 1)) * H * 4
            return b, 2.0 * T * K * F * H + 2.0 * T * Fs * H
        if kind == "router":
            return self.router + T * H * eb + T * (s.n_expert + (1 if Fs else 0)) * 4, 2.0 * T * H * s.n_expert
        if kind == "combine":
            return T * (K + 1) * H * 4 + T * H * 4, 0.0
        if kind == "gather":  # the routed rows (the shared expert reads x itself)
            return T * K * H * eb + T * H * eb, 0.0
        return None, None


def roofline_of(model, kind, T, d, avg_us, hbm, tc, tc_kind, workload):
    b, f = model.kernel(kind, T, d)
    if b is None or not avg_us:
        return {"kernel": kind, "bound": None, "achieved": None, "peak": None, "unit": None, "frac": None,
                "traffic": None}
    t = avg_us * 1e-6
    tensor = model.spec.dtype == "bf16" and f / (tc * 1e12) > b / (hbm * 1e9)
    if tensor:
        ach, peak, unit, bound, alg = f / t / 1e12, tc, "TFLOP/s", "tensor", f
    else:
        ach, peak, unit, bound, alg = b / t / 1e9, hbm, "GB/s", "hbm", b
    return {"kernel": kind, "bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
            "traffic": _traffic_from_profiles(kind, workload, T), "algorithmic_per_launch": alg,
            "avg_us": avg_us, "peak_kind": "hbm" if bound == "hbm" else tc_kind}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
_LINK_PEAK = {}


def host_link_peak(torch, dev):
    """GB/s of a pinned host -> device copy (the host link), measured once."""
    if dev in _LINK_PEAK:
        return _LINK_PEAK[dev]
    n = 512 << 20
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev)
    d.copy_(h, non_blocking=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 0.0
    # the best of three timings: a single one has read far low on one box
    for _ in range(3):
        e0.record(s)
        for _ in range(4):
            d.copy_(h, non_blocking=True)
        e1.record(s)
        torch.cuda.synchronize(dev)
        best = max(best, 4 * n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    _LINK_PEAK[dev] = best
    del h, d
    return _LINK_PEAK[dev]


class Runner:
    """One layer configuration on the GPU: n_layers layers with distinct weight
    memory, N_BATCHES token batches, and the measurements of a token count."""

    def __init__(self, spec, Tmax, n_layers, dev, dist, rank, sampler, peaks):
        import torch
        import sparse_mixture_experts_gb300 as moe
        self.torch, self.moe = torch, moe
        self.spec, self.Tmax, self.n_layers, self.dev, self.dist = spec, Tmax, n_layers, dev, dist
        self.sampler = sampler
        self.hbm, self.tc_burst, self.tc_sustained, self.peak_src = peaks
        self.model = Model(spec)
        self.w = synth.make_weights(spec, seed=0)
        wt = {}
        for k, v in self.w.items():
            t = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16 else \
                torch.from_numpy(v)
            wt[k] = t.to(dev)
        self.mxfp4 = spec.expert_format == "mxfp4"
        if self.mxfp4:  # the ABI takes the MXFP4 blocks in the gate_up_w / down_w slots
            wt["gate_up_w"] = wt.pop("gate_up_blocks")
            wt["down_w"] = wt.pop("down_blocks")
        self.q4 = spec.expert_format == "q4"
        if self.q4:  # and the Q4 records in the slots of the tensors they stand for
            for k in [k for k in wt if k.endswith("_q4")]:
                wt[k[:-3]] = wt.pop(k)
        cfg = moe.MoEConfig(
            hidden=spec.hidden, n_expert=spec.n_expert, top_k=spec.top_k, expert_ff=spec.expert_ff,
            shared_ff=spec.shared_ff,
            router_mode=moe.ROUTER_SOFTMAX_TOPK if spec.router_mode == "softmax_topk" else moe.ROUTER_TOPK_SOFTMAX,
            norm_topk_prob=spec.norm_topk_prob, weights_scale=spec.weights_scale,
            act=moe.ACT_SWIGLU if spec.act == "swiglu" else moe.ACT_CLAMP_GLU, act_alpha=spec.act_alpha,
            act_limit=spec.act_limit, has_bias=spec.has_bias, gate_up_interleaved=spec.gate_up_interleaved,
            w_dtype=moe.DT_MXFP4 if self.mxfp4 else moe.DT_Q4 if self.q4 else (
                moe.DT_BF16 if spec.dtype == "bf16" else moe.DT_F32),
            act_dtype=moe.DT_BF16 if spec.dtype == "bf16" else moe.DT_F32, out_dtype=moe.DT_F32, max_tokens=Tmax,
            resident_experts=spec.resident_experts)
        self.layers = [moe.MoELayer(cfg, wt, device=dev) for _ in range(n_layers)]
        del wt
        torch.cuda.empty_cache()
        self.x_np = synth.make_x(spec, Tmax * N_BATCHES, seed=1 + rank)
        self.xt = torch.from_numpy(self.x_np.view(np.int16)).view(torch.bfloat16) if self.x_np.dtype == np.uint16 \
            else torch.from_numpy(self.x_np)
        self.x_dev = self.xt.to(dev)
        self.out = torch.empty((Tmax, spec.hidden), dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def step(self, i, n_tok):
        b = (i % N_BATCHES) * self.Tmax
        self.layers[i % self.n_layers].forward(self.x_dev[b:b + n_tok], self.out[:n_tok], self.stream)

    def sync(self):
        self.torch.cuda.synchronize(self.dev)

    def timed(self, n_tok, K):
        """ms for exactly K steps between a barrier and a synchronize on both
        sides, CUDA events on the launching stream; max over ranks."""
        torch = self.torch
        barrier(self.dist)
        self.sync()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for i in range(K):
            self.step(i, n_tok)
        e1.record(self.stream)
        self.sync()
        ms = e0.elapsed_time(e1)
        barrier(self.dist)
        return reduce_max(ms, self.dist)

    def per_step_median(self, n_tok, K):
        """Median over K steps of each step's own event pair."""
        torch = self.torch
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
        self.sync()
        ev[0].record(self.stream)
        for i in range(K):
            self.step(i, n_tok)
            ev[i + 1].record(self.stream)
        self.sync()
        return statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(K))

    def keep_loaded(self, n_tok, seconds):
        end = time.time() + seconds
        i = 0
        while time.time() < end:
            self.step(i, n_tok)
            i += 1
            if i % 64 == 0:
                self.sync()
        self.sync()

    def routing_stats(self, n_tok, K):
        """Distinct experts per step (mean over the batches the K steps use),
        and the realised expert load of those batches."""
        distinct, loads = [], []
        for bi in range(N_BATCHES):
            b = bi * self.Tmax
            self.layers[0].forward(self.x_dev[b:b + n_tok], self.out[:n_tok], self.stream)
            c = self.layers[0].expert_counts(self.stream).cpu().numpy()
            distinct.append(int((c > 0).sum()))
            loads.append(c)
        used = [i % N_BATCHES for i in range(K)]
        d_avg = float(np.mean([distinct[b] for b in used]))
        c = loads[0]
        load = {"max_rows": int(c.max()), "min_rows": int(c.min()), "mean_rows": float(c.mean()),
                "max_over_mean": float(c.max() / max(c.mean(), 1e-9)), "experts_with_rows": int((c > 0).sum())}
        return d_avg, load

    def kernel_times(self, n_tok, K):
        for l in self.layers:
            l.timing_enable(K + 8)
        for j in range(K):
            self.step(j, n_tok)
        self.sync()
        kt = {}
        for l in self.layers:
            for k, (ms, n) in l.timing_read().items():
                a, b = kt.get(k, (0.0, 0))
                kt[k] = (a + ms, b + n)
            l.timing_enable(0)
        total = sum(ms for ms, _ in kt.values())
        return {k: {"avg_us": 1e3 * ms / n, "share": ms / total if total else None, "launches": n}
                for k, (ms, n) in kt.items() if n}

    def measure(self, n_tok, K, warmup, workload, load_s=0.5):
        """Everything the bench reports for one token count."""
        for i in range(max(3, warmup)):
            self.step(i, n_tok)
        self.sync()
        for l in self.layers:
            l.status()
        t0 = time.time()
        self.keep_loaded(n_tok, load_s)           # bring the clocks to their loaded state
        res0 = self.residency_totals()
        ms = self.timed(n_tok, K)
        res1 = self.residency_totals()
        t_timed = time.time()
        med = self.per_step_median(n_tok, max(K, MEDIAN_MIN_STEPS))
        self.keep_loaded(n_tok, 0.1)
        t1 = time.time()
        clocks = self.sampler.summary(t0, t1) if self.sampler else None
        launches = self.layers[(K - 1) % self.n_layers].last_launch_count
        kernels = self.kernel_times(n_tok, K)
        d_avg, load = self.routing_stats(n_tok, K)
        for l in self.layers:
            l.status()
        ws = self.dist.get_world_size() if self.dist is not None else 1
        mps = ms / K
        m = self.model
        sb, sf = m.step_bytes(n_tok, d_avg), m.step_flops(n_tok)
        # a dense GEMM held at the power cap runs at the sustained rate; else the burst one
        capped = bool(clocks and "sw_power_cap" in clocks.get("reasons", []))
        tc, tc_kind = (self.tc_sustained, "sustained") if capped and self.tc_sustained else (self.tc_burst, "burst")
        t_hbm, t_tc = sb / (self.hbm * 1e9), sf / (tc * 1e12)
        floor = max(t_hbm, t_tc) if self.spec.dtype == "bf16" else t_hbm
        if "experts" in kernels or "experts_mxfp4" in kernels or "experts_q4" in kernels:
            path = "weight-streaming tensor-core"
        elif "fused" in kernels:
            path = "fused"
        elif "gather" in kernels and "up" in kernels and "combine" in kernels and self.spec.dtype == "bf16":
            path = "tensor-core"
        else:
            path = "stream"
        top = max(kernels, key=lambda k: kernels[k]["avg_us"] * kernels[k]["launches"])
        residency = self.residency_summary(res0, res1, K, kernels)
        if top == "residency" and residency and residency["host_link_gbs"]:
            # the copies of the missing experts over the host link, against that link's
            # copy rate measured in this run
            peak = host_link_peak(self.torch, self.dev)
            roof = {"kernel": "residency", "bound": "host-link", "achieved": residency["host_link_gbs"],
                    "peak": peak, "unit": "GB/s", "frac": residency["host_link_gbs"] / peak, "traffic": None,
                    "algorithmic_per_launch": residency["host_bytes_per_step"], "avg_us": kernels[top]["avg_us"],
                    "peak_kind": "host-link", "peak_source": "pinned host -> device cudaMemcpyAsync, measured in this run"}
        else:
            roof = roofline_of(m, top, n_tok, d_avg, kernels[top]["avg_us"], self.hbm, tc, tc_kind, workload)
            roof["peak_source"] = self.peak_src
        return {
            "tokens": n_tok, "steps": K, "ms_per_step": mps, "ms_per_step_median": med,
            "median_steps": max(K, MEDIAN_MIN_STEPS), "tokens_per_s": ws * n_tok / (mps * 1e-3),
            "path": path, "distinct_experts": d_avg, "load": load,
            "step_roofline": {"bytes": sb, "flops": sf, "hbm_frac": t_hbm / (mps * 1e-3),
                              "tc_frac": t_tc / (mps * 1e-3) if self.spec.dtype == "bf16" else None,
                              "floor_us": floor * 1e6, "bound": "hbm" if floor == t_hbm else "tensor",
                              "frac_of_max_floor": floor / (mps * 1e-3), "tc_peak": tc, "tc_peak_kind": tc_kind},
            "roofline": roof, "kernels": kernels, "clocks": clocks, "gpu_launches_per_step": launches,
            "timed_region_s": t_timed - t0,
            "residency": residency,
        }

    def residency_totals(self):
        """Summed hit / miss / byte counters of the layers (expert residency)."""
        if not self.spec.resident_experts:
            return None
        tot = {"hits": 0, "misses": 0, "bytes": 0}
        for l in self.layers:
            _, st = l.residency()
            for k in tot:
                tot[k] += st[k]
        return tot

    def residency_summary(self, a, b, K, kernels):
        if a is None:
            return None
        d = {k: (b[k] - a[k]) / K for k in a}
        r = kernels.get("residency")
        us_step = r["avg_us"] * r["launches"] / K if r else None  # residency time per step
        return {"slots": self.spec.resident_experts, "hits_per_step": d["hits"], "misses_per_step": d["misses"],
                "host_bytes_per_step": d["bytes"],
                "host_link_gbs": (d["bytes"] / (us_step * 1e-6) / 1e9) if us_step and d["bytes"] else None,
                "note": "misses are copied from pinned host memory over the host link by the residency step"}

    def e2e(self, n_tok, K, warmup):
        """The metric through moe_forward_host: pinned host buffers, the copies
        in and out inside the timed region."""
        torch = self.torch
        x_host = self.xt[:self.Tmax * N_BATCHES].pin_memory()
        out_host = torch.empty((self.Tmax, self.spec.hidden), dtype=torch.float32).pin_memory()
        for j in range(max(3, warmup)):
            b = (j % N_BATCHES) * self.Tmax
            self.layers[j % self.n_layers].forward_host(x_host[b:b + n_tok], out_host[:n_tok], self.stream)
        self.sync()
        barrier(self.dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for j in range(K):
            b = (j % N_BATCHES) * self.Tmax
            self.layers[j % self.n_layers].forward_host(x_host[b:b + n_tok], out_host[:n_tok], self.stream)
        e1.record(self.stream)
        self.sync()
        ms = reduce_max(e0.elapsed_time(e1), self.dist)
        for l in self.layers:
            l.status()
        ws = self.dist.get_world_size() if self.dist is not None else 1
        eb = 2 if self.spec.dtype == "bf16" else 4
        return {"value": ws * n_tok * K / (ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": n_tok * self.spec.hidden * eb, "d2h_bytes_per_step": n_tok * self.spec.hidden * 4}

    def l2_note(self):
        gb = self.layers[0].device_bytes * self.n_layers / 1e9
        if self.n_layers == 1:
            return f"one layer ({gb:.3f} GB): fits L2; a latency-bound case"
        return f"inputs larger than L2: steps rotate over {self.n_layers} layers with distinct weight memory ({gb:.1f} GB)"

    def close(self):
        for l in self.layers:
            l.close()
        self.layers = []
        del self.x_dev, self.out
        self.torch.cuda.empty_cache()


def run_ours(args, spec, T, extra_T, n_layers, workload):
    import torch
    from sparse_mixture_experts_gb300 import build as libbuild

    ws, rank, local = dist_env()
    dist = dist_init(ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not libbuild.up_to_date():
        if rank == 0:
            libbuild.build()
        barrier(dist)
    peaks = _peaks()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)

    # ---- headline workload ----
    Tmax = max((T,) + tuple(extra_T))
    run = Runner(spec, Tmax, n_layers, dev, dist, rank, sampler, peaks)
    head = run.measure(T, args.steps, args.warmup, workload, load_s=1.0)
    extra = {str(n): run.measure(n, args.steps, args.warmup, workload) for n in extra_T}
    e2e = run.e2e(T, args.steps, args.warmup)
    l2 = run.l2_note()
    w_head = run.w
    run.close()
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baselines(spec, w_head, args.cpu_budget, args.cpu_budget / 4)

    # ---- every configuration at its full sizes ----
    workloads = {}
    if not args.no_workloads:
        for name, (wspec, counts, nl) in SWEEP.items():
            if HEADLINE_SWEEP.get(workload) == name:
                entries = {str(n): e for n, e in [(T, head)] + [(int(k), v) for k, v in extra.items()]}
                workloads[name] = {"config": wspec.name, "layers_rotated": n_layers, "l2": l2,
                                   "tokens": dict(sorted(entries.items(), key=lambda kv: int(kv[0]))),
                                   "cpu_baseline": cpu}
                continue
            r = Runner(wspec, max(counts), nl, dev, dist, rank, sampler, peaks)
            entries = {str(n): r.measure(n, args.steps, args.warmup, name) for n in counts}
            note = r.l2_note()
            wsw = r.w
            r.close()
            wcpu = None
            if rank == 0 and ws == 1 and not args.no_cpu_baseline:
                wcpu = cpu_baselines(wspec, wsw, args.cpu_budget / 3, args.cpu_budget / 8)
            workloads[name] = {"config": wspec.name, "layers_rotated": nl, "l2": note, "tokens": entries,
                               "cpu_baseline": wcpu}
    sampler.stop()

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["tokens_per_s"], "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": _spec_dtype(spec), "data": "synthetic",
            "config": {"workload": f"{spec.name}, {T} tokens per step", "tokens_per_step": T,
                       "layers_rotated": n_layers, "l2": l2, "token_batches": N_BATCHES,
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "distinct_experts_per_step": head["distinct_experts"], "path": head["path"]},
            "roofline": head["roofline"],
            "step_roofline": head["step_roofline"],
            "ms_per_step_median": head["ms_per_step_median"],
            "kernels": head["kernels"],
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": head["gpu_launches_per_step"] * args.steps,
            "clocks": head["clocks"],
            "other_token_counts": {k: {"tokens_per_s": v["tokens_per_s"], "ms_per_step": v["ms_per_step"], "kernels": v["kernels"],
                                       "distinct_experts": v["distinct_experts"],
                                       "hbm_frac": v["step_roofline"]["hbm_frac"],
                                       "roofline": v["roofline"], "residency": v["residency"]}
                                   for k, v in extra.items()},
            "workloads": workloads,
        }
        if head["residency"]:
            line["residency"] = head["residency"]
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
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
    ap.add_argument("--no-workloads", action="store_true", help="measure the headline workload only")
    ap.add_argument("--check-launch", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "ours" and check_world(args.gpus) == "spawn":
        return subprocess.call(launcher_cmd(args.gpus, argv))
    if args.check_launch:
        return run_check_launch()
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
