"""Benchmark: Qwen3-style decoder prefill throughput and decode-step latency on one GB300 (per process),
through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

The default workload is the largest single-GPU one: the Qwen3-8B shape, causal prefill of 1 x 32768
tokens, then decode of 16 sequences at a 32,768-token pre-filled context (77 GB bf16 cache).
A step is one causal prefill (embedding, all layers, final norm, LM head on each sequence's last row)
of the workload's batch of synthetic token ids, on random-init bf16 weights of the named shape, and its
greedy token; the `decode` block times greedy decode steps (each step's argmax fed back). With
N > 1 (torchrun, one process per GPU) every rank runs an independent replica ("replicas only": the
forward pass has no exchange step); value = all ranks' tokens / the slowest rank's time.

Prints one JSON line. ``value`` is device-timed (CUDA events, inputs resident in HBM); ``e2e`` times the
same step through qwen3_prefill_host with pinned host buffers (ids host->device and logits
device->host inside the timed region). ``roofline`` is for the kernel class with the largest share of
the timed region, from per-launch CUDA events recorded by the library on the launch stream.
``cpu_baseline`` / ``--impl reference`` time the oracle (single-threaded C++) on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s and decode-step ms on 1 GB300; % of bf16-tensor / HBM roofline"
DEFAULT_WORKLOAD = "8b-prefill-1x32768-decode-16@32768"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ----------------------------------------------------------------------------- algorithmic work

def kernel_work(cfg: dict, B: int, T: int) -> dict:
    """Algorithmic FLOPs (tensor-bound classes) or bytes (memory-bound classes) of ONE launch of each
    kernel class in a prefill of B x T starting at length 0. Causal attention counts the T(T+1)/2
    visible query/key pairs: 4 * dh FLOPs per pair and query head (QK^T and PV)."""
    d, dh, F, V = cfg["hidden"], cfg["head_dim"], cfg["intermediate"], cfg["vocab"]
    hq, hkv = cfg["n_q_heads"], cfg["n_kv_heads"]
    M = B * T
    qkv_n = (hq + 2 * hkv) * dh
    return {
        "gemm_qkv_norm_rope_append": ("tensor", 2.0 * M * qkv_n * d),
        "gemm_o_residual": ("tensor", 2.0 * M * d * hq * dh),
        "gemm_gateup_swiglu": ("tensor", 2.0 * M * 2 * F * d),
        "gemm_down_residual": ("tensor", 2.0 * M * d * F),
        "gemm_lmhead": ("tensor", 2.0 * B * V * d),
        "attn_prefill": ("tensor", 4.0 * B * hq * dh * T * (T + 1) / 2),
        "rmsnorm": ("hbm", 2.0 * M * d * 2),
        "qknorm_rope_append": ("hbm", 2.0 * M * qkv_n * 2),
        "embed": ("hbm", 2.0 * M * d * 2),
    }


def step_flops(cfg: dict, B: int, T: int) -> float:
    w = kernel_work(cfg, B, T)
    L = cfg["n_layers"]
    per_layer = sum(w[k][1] for k in ("gemm_qkv_norm_rope_append", "gemm_o_residual", "gemm_gateup_swiglu",
                                       "gemm_down_residual", "attn_prefill"))
    return L * per_layer + w["gemm_lmhead"][1]


# ----------------------------------------------------------------------------- profiles

def traffic_from_profiles(kernel_class: str, workload: str):
    """Per-launch DRAM bytes of a kernel class from a committed ncu summary, or None when no summary
    exists or the kernel source changed after the counters were taken (source hash recorded)."""
    src = {"gemm": "gemm.cu", "attn": "attention.cu"}.get(kernel_class.split("_")[0], "kernels.cu")
    path = os.path.join(ROOT, "profiles", f"{kernel_class}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(os.path.join(ROOT, "qwen3_decoder_transformer_gb300", "csrc", src), "rb").read())
    if cur.hexdigest()[:16] != h.group(1)[:16]:
        return None
    return float(m.group(1))


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.25)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
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
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over the process group (identity when not distributed)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- oracle baseline

def cpu_description() -> dict:
    """Host cores and CPU model of this machine (for the baseline's record)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                k, _, v = ln.partition(":")
                k = k.strip().lower()
                if k in ("model name", "cpu model", "hardware") and v.strip():
                    model = v.strip()
                    break
                if k == "cpu part" and model is None:
                    model = "cpu part " + v.strip()
    except OSError:
        pass
    if model is None or model.startswith("cpu part"):
        try:  # lscpu names Arm cores that /proc/cpuinfo lists only by part number
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for ln in out.splitlines():
                if ln.lower().startswith("model name:"):
                    model = ln.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or platform.machine(),
            "machine": platform.machine()}


class OracleBench:
    """The oracle (single-threaded C++, as it stands) timed on a bounded sample of the workload: one
    decoder layer (steps a2-a9) of the workload's shape over a prefix of `tokens` rows, extrapolated to
    the workload's whole prefill step by the ratio of algorithmic FLOPs. A whole step is far beyond a
    bounded run (the 8B 1x32768 prefill is 7.7e14 FLOPs; the oracle runs a few GFLOP/s)."""

    def __init__(self, cfg: dict, seed: int):
        import oracle as O
        from qwen3_decoder_transformer_gb300 import synth
        self.O = O
        self.cfg = cfg
        d = cfg["hidden"]
        w = {"embed": None, "lm_head": None, "final_norm": synth._gain(d, synth._seed(seed, "final_norm"), "cpu")}
        for name in synth.LAYER_NAMES:
            w[name] = [None] * cfg["n_layers"]
        for name, t in synth.make_layer(cfg, seed, 0).items():
            w[name][0] = t
        self.model = O.Model(cfg, synth.weights_to_numpy(w))
        # layer-0 inputs: rows distributed as embedding rows (bf16 N(0, 0.02)), 1024 at most
        self.x = synth.to_numpy_bits(synth._normal((1024, d), 0.02, synth._seed(seed, "bench_rows"), "cpu"))

    def run(self, tokens: int) -> float:
        """Seconds for layer 0 (norm, Q/K/V + q/k-norm + RoPE, causal GQA attention, o_proj + residual,
        norm, SwiGLU MLP, down + residual) over `tokens` rows at positions 0..tokens-1."""
        c = self.cfg
        tokens = min(tokens, self.x.shape[0])
        x = self.x[:tokens]
        pos = np.arange(tokens, dtype=np.int32)
        kc = np.zeros((1, c["n_kv_heads"], tokens, c["head_dim"]), dtype=np.uint16)
        vc = np.zeros_like(kc)
        t0 = time.perf_counter()
        q, k, v = self.model.layer_qkv(0, x, pos)
        kc[0] = k.transpose(1, 0, 2)
        vc[0] = v.transpose(1, 0, 2)
        self.model.layer_out(0, x, q, pos, kc, vc, np.zeros(tokens, dtype=np.int32))
        return time.perf_counter() - t0

    @staticmethod
    def layer_flops(cfg: dict, tokens: int) -> float:
        d, dh, F = cfg["hidden"], cfg["head_dim"], cfg["intermediate"]
        hq, hkv = cfg["n_q_heads"], cfg["n_kv_heads"]
        gemm = 2.0 * tokens * (d * (hq + 2 * hkv) * dh + hq * dh * d + 3 * d * F)
        return gemm + 4.0 * hq * dh * tokens * (tokens + 1) / 2

    def extrapolate(self, seconds: float, tokens: int, B: int, T: int) -> float:
        """Workload tokens/s implied by `seconds` for one layer over `tokens` rows."""
        step_s = seconds * step_flops(self.cfg, B, T) / self.layer_flops(self.cfg, tokens)
        return B * T / step_s

    def describe(self, tokens: int, B: int, T: int) -> str:
        ratio = step_flops(self.cfg, B, T) / self.layer_flops(self.cfg, tokens)
        return (f"extrapolated: oracle (single-threaded C++, fp64 accumulation, bf16 emulation) timed on one "
                f"decoder layer of the workload's shape over a {tokens}-token prefix, scaled by the FLOP ratio "
                f"{ratio:.4g} to the {B}x{T} prefill step ({self.cfg['n_layers']} layers, causal attention, "
                f"LM head on the last rows); tokens/s = {B * T} / extrapolated step time")


def sample_tokens(cfg: dict, budget_flops: float) -> int:
    """Prefix length whose one-layer oracle pass costs about `budget_flops` (the oracle runs a few
    GFLOP/s on one core)."""
    per_tok = OracleBench.layer_flops(cfg, 1)
    return int(max(2, min(1024, budget_flops / per_tok)))


# ----------------------------------------------------------------------------- arms

def run_reference(args, wl):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    cfg = wl["model"]
    B, T = wl["prefill"]
    ob = OracleBench(cfg, wl["seed"])
    # whole run about 2-3 minutes of single-core work: ~2e11 FLOPs shared by the timed steps
    toks = sample_tokens(cfg, 2e11 / max(1, args.steps))
    for _ in range(args.warmup):
        ob.run(2)
    times = [ob.run(toks) for _ in range(args.steps)]
    sec = sum(times) / len(times)
    v = ob.extrapolate(sec, toks, B, T)
    desc = ob.describe(toks, B, T)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * B * T / v,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate/bf16-storage",
            "data": "synthetic (random-init weights, uniform token ids)",
            "config": {"workload": args.workload, "batch": B, "seq_len": T,
                       "sample": f"one layer over a {toks}-token prefix per step, {1e3 * sec:.0f} ms each"},
            "cpu_baseline": dict({"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc},
                                 **cpu_description()),
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, wl):
    import torch

    from qwen3_decoder_transformer_gb300 import binding, build, synth
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    build.build()
    cfg = wl["model"]
    B, T = wl["prefill"]
    V = cfg["vocab"]
    dev = torch.device("cuda", local)
    w = synth.make_weights(cfg, wl["seed"], device=dev)
    ids = synth.make_ids(V, B, T, wl["seed"], device=dev)
    m = binding.Model(cfg, w, max_batch=B, capacity=T, max_tokens=B * T)
    logits = torch.empty(B, V, dtype=torch.float32, device=dev)
    next_ids = torch.empty(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():  # prefill, then the greedy next token of every sequence
        m.set_length(0, 0)
        m.prefill(ids, logits)
        binding.op_greedy(logits, next_ids)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if m.get_error() != 0:
        raise RuntimeError("device error flag set during warm-up")

    # ---- device-timed region: the headline value, no per-launch instrumentation
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    elapsed_ms = start.elapsed_time(stop)
    rc = m.get_error()
    if rc != 0:
        raise RuntimeError(f"device error flag {rc} in the timed region")
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    value = world * B * T * args.steps / (elapsed_ms / 1e3)

    # ---- same K steps again with per-launch CUDA events recorded by the library on this stream
    m.set_timing(True)
    m.kernel_times()  # reset
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_stop.record(stream)
    torch.cuda.synchronize()
    instrumented_ms = t_start.elapsed_time(t_stop)
    kt = m.kernel_times()
    m.set_timing(False)

    # ---- end-to-end through the host-buffer entry point
    h_ids = torch.empty(B, T, dtype=torch.int32, pin_memory=True)
    h_ids.copy_(ids.cpu())
    h_logits = torch.empty(B, V, dtype=torch.float32, pin_memory=True)
    for _ in range(max(1, args.warmup)):
        m.set_length(0, 0)
        m.prefill_host(h_ids.numpy(), h_logits.numpy())
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        m.set_length(0, 0)
        m.prefill_host(h_ids.numpy(), h_logits.numpy())
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e = {"value": world * B * T * args.steps / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": B * T * 4, "d2h_bytes_per_step": B * V * 4}

    # ---- roofline of the dominant kernel class
    peaks, peak_src = load_peaks()
    work = kernel_work(cfg, B, T)
    per_kernel = {k: {"ms_per_step": v[0] / args.steps, "launches_per_step": v[1] / args.steps,
                      "share": v[0] / max(1e-9, sum(x[0] for x in kt.values()))} for k, v in kt.items() if v[1]}
    dom = max((k for k in per_kernel if k in work), key=lambda k: kt[k][0])
    bound, units = work[dom]
    avg_ms = kt[dom][0] / kt[dom][1]
    long_region = instrumented_ms > 1000.0
    if bound == "tensor":
        achieved = units / (avg_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
        unit = "TFLOP/s"
    else:
        achieved = units / (avg_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    traffic = traffic_from_profiles(dom, args.workload)
    roof = {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic,
            "peak_source": f"{peak_src} ({'sustained' if (bound == 'tensor' and long_region) else 'burst'})",
            "algorithmic_per_launch": units, "avg_launch_ms": avg_ms}
    step_tf = step_flops(cfg, B, T)
    # the tensor-core share of the step: GEMM + attention FLOPs over the time those kernels took
    tensor_classes = [k for k, v in work.items() if v[0] == "tensor" and k in kt and kt[k][1]]
    ga_flops = sum(work[k][1] * kt[k][1] for k in tensor_classes)
    ga_ms = sum(kt[k][0] for k in tensor_classes)
    ga_peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    gemm_attn = {"tflops": ga_flops / (ga_ms / 1e3) / 1e12, "peak": ga_peak,
                 "frac": ga_flops / (ga_ms / 1e3) / 1e12 / ga_peak, "ms_per_step": ga_ms / args.steps,
                 "peak_source": f"{peak_src} ({'sustained' if long_region else 'burst'})",
                 "classes": tensor_classes}
    launches = m.launch_count(B, T) + 2  # + the length reset before each step and the greedy kernel
    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random-init bf16 weights N(0,0.02), gains 1+U(-0.1,0.1), uniform token ids)",
            "config": {"workload": args.workload, "batch": B, "seq_len": T, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2: each step streams all weights (%.2f GB) through HBM"
                             % (sum(t.numel() * 2 for k, t in _flat(w)) / 1e9)},
            "e2e": e2e, "gpu_launches": launches * args.steps,
            "roofline": roof,
            "step_tflops": step_tf / 1e12,
            "step_frac_of_peak": {"burst": step_tf / (elapsed_ms / args.steps / 1e3) / 1e12 / peaks["bf16_tflops"],
                                  "sustained": step_tf / (elapsed_ms / args.steps / 1e3) / 1e12
                                  / peaks["bf16_tflops_sustained"]},
            "gemm_attention_frac_of_peak": gemm_attn,
            "clocks": clk.summary(), "kernels": per_kernel,
            "kernels_note": "per-kernel times from a second run of the same steps with a CUDA event pair around "
                            "every launch (%.3f ms/step with events vs %.3f without)"
                            % (instrumented_ms / args.steps, elapsed_ms / args.steps)}
    if wl["decode_steps"] > 0:
        m.close()
        line["decode"] = measure_decode(binding, synth, torch, cfg, wl, w, dev, args.decode_steps)
        peaks_hbm = peaks["hbm_gbs"]
        line["decode"]["attention_roofline"]["peak"] = peaks_hbm
        line["decode"]["attention_roofline"]["frac"] = line["decode"]["attention_roofline"]["achieved"] / peaks_hbm
        line["decode"]["step_hbm_frac"] = line["decode"]["step_hbm_gbs"] / peaks_hbm
    if world == 1 and not args.no_cpu_baseline:
        ob = OracleBench(cfg, wl["seed"])
        toks = sample_tokens(cfg, 2.5e10)
        dt = ob.run(toks)
        line["cpu_baseline"] = dict({"value": ob.extrapolate(dt, toks, B, T), "unit": "tokens/s", "cores": 1,
                                     "kind": "oracle", "sample": ob.describe(toks, B, T), "seconds": dt},
                                    **cpu_description())
    print(json.dumps(line), flush=True)
    m.close()


def measure_decode(binding, synth, torch, cfg, wl, w, dev, steps_cap: int):
    """Decode-step latency at the workload's pre-filled context, through qwen3_decode_step (graph replay).
    The cache holds bf16 N(0,1) K/V for the first `ctx` positions of every sequence."""
    Bd, ctx = wl["decode_batch"], wl["prefilled_ctx"]
    steps = min(wl["decode_steps"], steps_cap)
    L, V, Hkv, dh = cfg["n_layers"], cfg["vocab"], cfg["n_kv_heads"], cfg["head_dim"]
    m = binding.Model(cfg, w, max_batch=Bd, capacity=ctx + wl["decode_steps"], max_tokens=max(Bd, 128))
    for layer in range(L):
        k, v = m.kv_view(layer)
        shape = (Bd, Hkv, ctx, dh)
        k[:, :, :ctx].copy_(synth.make_kv_normal(shape, wl["seed"], layer, "k", device=dev))
        v[:, :, :ctx].copy_(synth.make_kv_normal(shape, wl["seed"], layer, "v", device=dev))
    ids = synth.make_ids(V, Bd, 1, wl["seed"] + 100, device=dev).reshape(Bd)
    first = ids.clone()
    logits = torch.empty(Bd, V, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):  # warm-up (the first call captures the graph)
        m.set_length(ctx, Bd)
        m.decode_step(ids, logits)
        binding.op_greedy(logits, ids)
    torch.cuda.synchronize()
    m.set_length(ctx, Bd)
    ids.copy_(first)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):  # greedy generation: each step's argmax is the next step's input
        m.decode_step(ids, logits)
        binding.op_greedy(logits, ids)
    b.record(stream)
    torch.cuda.synchronize()
    if m.get_error() != 0:
        raise RuntimeError("device error flag set during decode")
    ms = a.elapsed_time(b) / steps
    # per-kernel breakdown: the same steps, eager, with per-launch events
    m.set_length(ctx, Bd)
    m.set_timing(True)
    m.kernel_times()
    for _ in range(steps):
        m.decode_step(ids, logits)
    kt = m.kernel_times()
    m.set_timing(False)
    kv_bytes = 2.0 * Bd * Hkv * dh * 2 * (ctx + (steps + 1) / 2.0)  # K and V read per layer, mean context
    att_ms = kt["attn_decode"][0] / kt["attn_decode"][1] * 2  # two launches (split + merge) per timed pair
    w_bytes = float(sum(t.numel() * 2 for _, t in _flat(w)))
    out = {"batch": Bd, "context": ctx, "steps": steps, "ms_per_step": ms,
           "kernels": {k: {"ms_per_step": v[0] / steps, "launches_per_step": v[1] / steps}
                       for k, v in kt.items() if v[1]},
           "attention_roofline": {"bound": "hbm", "achieved": kv_bytes / (att_ms / 1e3) / 1e9,
                                  "unit": "GB/s", "algorithmic_bytes_per_launch": kv_bytes,
                                  "avg_launch_ms": att_ms},
           "step_hbm_gbs": (w_bytes + L * kv_bytes) / (ms / 1e3) / 1e9}
    m.close()
    return out


def run_op(args, wl):
    """Time one kernel alone through its single-operation C entry point at the workload's shapes
    (small device footprint, for ncu captures and isolated roofline numbers)."""
    import torch

    from qwen3_decoder_transformer_gb300 import binding, build
    build.build()
    torch.cuda.set_device(0)
    cfg = wl["model"]
    B, T = wl["prefill"]
    d, dh, F, V = cfg["hidden"], cfg["head_dim"], cfg["intermediate"], cfg["vocab"]
    hq, hkv = cfg["n_q_heads"], cfg["n_kv_heads"]
    g = torch.Generator(device="cuda")
    g.manual_seed(wl["seed"])
    rnd = lambda *shape: torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)
    len0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    M = B * T
    if args.op == "attn_prefill":
        if args.rows:  # a prefill chunk of `rows` tokens after `len0` cached ones
            T, M = args.rows, B * args.rows
        len0.fill_(args.len0)
        q, kc, vc = rnd(B, hq, T, dh), rnd(B, hkv, T + args.len0, dh), rnd(B, hkv, T + args.len0, dh)
        out = torch.empty(M, hq * dh, dtype=torch.bfloat16, device="cuda")
        split, chunks = args.kv_split, max(1, args.kv_chunks)
        ws = torch.zeros(max(1, binding.attention_prefill_workspace(B, T, hq, hkv, dh, chunks) // 4),
                         dtype=torch.float32, device="cuda")
        fn = lambda: binding.op_attention_prefill(q, kc, vc, len0, out, kv_split=split, kv_chunks=chunks, work=ws,
                                                  heads_per_cta=args.heads)
        work, unit, bound = 4.0 * B * hq * dh * (T * (T + 1) / 2 + T * args.len0), "TFLOP/s", "tensor"
    elif args.op == "attn_decode":
        Bd, ctx = args.rows or wl["decode_batch"] or 16, wl["prefilled_ctx"] or T
        q, kc, vc = rnd(Bd, hq, dh), rnd(Bd, hkv, ctx + 8, dh), rnd(Bd, hkv, ctx + 8, dh)
        len0.fill_(ctx - 1)
        ws = torch.zeros(binding.attention_decode_workspace(Bd, hq, dh, ctx + 8) // 4, dtype=torch.float32,
                         device="cuda")
        out = torch.empty(Bd, hq * dh, dtype=torch.bfloat16, device="cuda")
        fn = lambda: binding.op_attention_decode(q, kc, vc, len0, ws, out)
        work, unit, bound = 2.0 * Bd * hkv * ctx * dh * 2, "GB/s", "hbm"
    elif args.op in ("gemm_gateup", "gemm_qkv", "gemm_o", "gemm_down"):
        N, K, epi = {"gemm_gateup": (2 * F, d, binding.EPI_SWIGLU), "gemm_qkv": ((hq + 2 * hkv) * dh, d, binding.EPI_BF16),
                     "gemm_o": (d, hq * dh, binding.EPI_RESIDUAL), "gemm_down": (d, F, binding.EPI_RESIDUAL)}[args.op]
        Mx = args.rows or M
        act, wt = rnd(Mx, K), rnd(N, K)
        c = torch.empty(Mx, N // 2 if epi == binding.EPI_SWIGLU else N, dtype=torch.bfloat16, device="cuda")
        fn = lambda: binding.op_gemm(act, wt, epi, c, R=c if epi == binding.EPI_RESIDUAL else None)
        work, unit, bound = 2.0 * Mx * N * K, "TFLOP/s", "tensor"
        if Mx <= 256:
            work, unit, bound = 2.0 * N * K + 2.0 * Mx * K + 2.0 * Mx * c.shape[1], "GB/s", "hbm"
    elif args.op == "qknorm_rope":
        H = hq + 2 * hkv
        qkv = rnd(M, H * dh)
        table = torch.empty(T, dh, dtype=torch.bfloat16, device="cuda")
        binding.op_rope_table(cfg["rope_theta"], dh, T, table)
        gq, gk = rnd(dh), rnd(dh)
        qo = torch.empty(B, hq, T, dh, dtype=torch.bfloat16, device="cuda")
        kc, vc = torch.empty(B, hkv, T, dh, dtype=torch.bfloat16, device="cuda"), torch.empty(
            B, hkv, T, dh, dtype=torch.bfloat16, device="cuda")
        fn = lambda: binding.op_qknorm_rope_append(qkv, B, T, hq, hkv, dh, gq, gk, table, len0, 1e-6, qo, kc, vc)
        work, unit, bound = 2.0 * M * H * dh * 2, "GB/s", "hbm"
    elif args.op == "rmsnorm":
        Mx = args.rows or M
        x, gm = rnd(Mx, d), rnd(d)
        y = torch.empty_like(x)
        fn = lambda: binding.op_rmsnorm(x, gm, 1e-6, y)
        work, unit, bound = 2.0 * Mx * d * 2, "GB/s", "hbm"
    elif args.op == "embed":
        Mx = args.rows or M
        E = rnd(V, d)
        ids = torch.randint(0, V, (Mx,), generator=g, device="cuda", dtype=torch.int64).to(torch.int32)
        out = torch.empty(Mx, d, dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        fn = lambda: binding.op_embed(E, ids, out, err)
        work, unit, bound = 2.0 * Mx * d * 2, "GB/s", "hbm"
    elif args.op == "greedy":
        Bx = args.rows or wl["decode_batch"] or B
        logits = torch.randn(Bx, V, generator=g, device="cuda")
        nxt = torch.empty(Bx, dtype=torch.int32, device="cuda")
        fn = lambda: binding.op_greedy(logits, nxt)
        work, unit, bound = 4.0 * Bx * V, "GB/s", "hbm"
    elif args.op == "gemm_o_norm":  # o_proj (or down_proj with --rows) + residual fused with the next RMSNorm
        Mx = args.rows or M
        K = hq * dh
        act, wt, gm = rnd(Mx, K), rnd(d, K), rnd(d)
        x, y = rnd(Mx, d), torch.empty(Mx, d, dtype=torch.bfloat16, device="cuda")
        part = torch.zeros(binding.gemm_norm_part_floats(Mx), dtype=torch.float32, device="cuda")
        fn = lambda: binding.op_gemm_residual_norm(act, wt, x, gm, 1e-6, y, part)
        work, unit, bound = 2.0 * Mx * d * K, "TFLOP/s", "tensor"
    elif args.op == "decode_step":  # whole greedy decode steps (graph replay) at the workload's context
        cfgd = dict(cfg, n_layers=args.layers) if args.layers else cfg
        Bd = args.rows or wl["decode_batch"] or 1
        ctx = args.len0 or wl["prefilled_ctx"] or 1024
        from qwen3_decoder_transformer_gb300 import synth
        w = synth.make_weights(cfgd, wl["seed"], device="cuda")
        m = binding.Model(cfgd, w, max_batch=Bd, capacity=ctx + args.steps + args.warmup + 8, max_tokens=max(Bd, 128))
        Hkv_, dh_ = cfgd["n_kv_heads"], cfgd["head_dim"]
        for layer in range(cfgd["n_layers"]):
            k, v = m.kv_view(layer)
            k[:, :, :ctx].copy_(synth.make_kv_normal((Bd, Hkv_, ctx, dh_), wl["seed"], layer, "k", device="cuda"))
            v[:, :, :ctx].copy_(synth.make_kv_normal((Bd, Hkv_, ctx, dh_), wl["seed"], layer, "v", device="cuda"))
        m.set_length(ctx, Bd)
        ids = synth.make_ids(V, Bd, 1, wl["seed"] + 100, device="cuda").reshape(Bd)
        logits = torch.empty(Bd, V, dtype=torch.float32, device="cuda")

        def fn():
            m.decode_step(ids, logits)
            binding.op_greedy(logits, ids)
        wbytes = float(sum(t.numel() * 2 for _, t in _flat(w)))
        kvb = 2.0 * cfgd["n_layers"] * Bd * Hkv_ * dh_ * 2 * ctx
        work, unit, bound = wbytes + kvb, "GB/s", "hbm"
    else:
        raise SystemExit(f"unknown op {args.op}")
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.steps):
        fn()
    ev1.record()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / args.steps
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    peaks, src = load_peaks()
    peak = peaks["bf16_tflops"] if unit == "TFLOP/s" else peaks["hbm_gbs"]
    ach = work / (ms / 1e3) / scale
    print(json.dumps({"op": args.op, "workload": args.workload, "ms_per_launch": ms, "bound": bound,
                      "achieved": ach, "unit": unit, "peak": peak, "frac": ach / peak,
                      "algorithmic_per_launch": work, "peak_source": src + " (burst)"}), flush=True)


# ----------------------------------------------------------------------------- generation features

def _timed(torch, fn, steps: int, warmup: int) -> float:
    """Mean ms of fn() over `steps` calls after `warmup` calls, CUDA events on the current stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def _kernel_split(m, fn, steps: int) -> dict:
    m.set_timing(True)
    m.kernel_times()
    for _ in range(steps):
        fn()
    kt = m.kernel_times()
    m.set_timing(False)
    return {k: round(v[0] / steps, 4) for k, v in kt.items() if v[1]}


def run_feature(args):
    """Time one generation feature on its own synthetic workload (one GPU; prints one JSON line):

    padded  left-padded batch ("A modern architecture: Qwen3", generation with a batch of prompts):
            Qwen3-0.6B shape, 32 prompts of 512..2048 tokens padded to 2048; prefill + greedy token,
            then 64 greedy decode steps (each step's argmax fed back).
    prefix  shared prefix (section 8): a 2048-token start shared by 32 prompts of 64..256 tokens;
            prefill of the start once + share + padded prefill of the prompts, against one padded
            prefill of the 32 concatenated prompts.
    window  sliding window (section 7): Qwen3-8B shape with a 4096-token window; decode of 16 sequences
            at position 32768 from a rolling buffer, and a banded 1 x 32768 prefill over a full cache.
    """
    import torch

    from qwen3_decoder_transformer_gb300 import binding, build, configs, synth
    build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks, src = load_peaks()
    K, Wm = args.steps, args.warmup
    line = {"feature": args.feature, "data": "synthetic (random-init bf16 weights, uniform token ids)",
            "peak_source": src}
    with ClockSampler(0) as clk:
        if args.feature in ("padded", "prefix"):
            cfg = configs.QWEN3_0P6B
            V = cfg["vocab"]
            seed = 5 if args.feature == "padded" else 6
            w = synth.make_weights(cfg, seed, device=dev)
            rng = np.random.default_rng(seed)
            pad_id = 151643 % V
        if args.feature == "padded":
            B, T, D = 32, 2048, 64
            real = rng.integers(512, T + 1, size=B)
            ids = synth.make_ids(V, B, T, seed, device=dev)
            for b in range(B):
                ids[b, :T - int(real[b])] = pad_id
            m = binding.Model(cfg, w, max_batch=B, capacity=T + D + 8, max_tokens=B * T)
            logits = torch.empty(B, V, dtype=torch.float32, device=dev)
            nxt = torch.empty(B, dtype=torch.int32, device=dev)

            def prefill():
                m.set_length(0, 0)
                m.prefill_padded(ids, real, logits)
                binding.op_greedy(logits, nxt)

            ms = _timed(torch, prefill, K, Wm)
            kern = _kernel_split(m, prefill, max(1, K // 4))
            work = kernel_work(cfg, B, T)
            att_ms = kern.get("attn_prefill", 0) / cfg["n_layers"]
            line.update({"batch": B, "width": T, "real_tokens": int(real.sum()), "prefill_ms": ms,
                         "real_tokens_per_s": float(real.sum()) / (ms / 1e3), "padded_tokens_per_s": B * T / (ms / 1e3),
                         "prefill_kernels_ms": kern,
                         "attn_prefill_frac_of_peak": work["attn_prefill"][1] / (att_ms / 1e3) / 1e12
                         / peaks["bf16_tflops"] if att_ms else None})
            prefill()

            def decode():
                m.decode_step(nxt, logits)
                binding.op_greedy(logits, nxt)

            line.update({"decode_steps": D, "decode_ms_per_step": _timed(torch, decode, D, 3)})
            assert m.get_error() == 0
            m.close()
        elif args.feature == "prefix":
            B, P, lo, hi = 32, 2048, 64, 256
            lens = rng.integers(lo, hi + 1, size=B)
            Tp = int(lens.max())
            pre = synth.make_ids(V, 1, P, seed, device=dev)
            body = synth.make_ids(V, B, Tp, seed + 1, device=dev)
            for b in range(B):
                body[b, :Tp - int(lens[b])] = pad_id
            full = torch.cat([pre.expand(B, P), body], dim=1).contiguous()
            for b in range(B):  # concatenated prompts, left-padded as a whole
                n = P + int(lens[b])
                full[b] = torch.cat([torch.full((P + Tp - n,), pad_id, dtype=torch.int32, device=dev),
                                     pre[0], body[b, Tp - int(lens[b]):]])
            m = binding.Model(cfg, w, max_batch=B, capacity=P + Tp + 8, max_tokens=B * (P + Tp))
            l1 = torch.empty(1, V, dtype=torch.float32, device=dev)
            la = torch.empty(B, V, dtype=torch.float32, device=dev)
            lb = torch.empty(B, V, dtype=torch.float32, device=dev)
            na = torch.empty(B, dtype=torch.int32, device=dev)
            nb = torch.empty(B, dtype=torch.int32, device=dev)

            def shared():
                m.set_length(0, 0)
                m.prefill(pre, l1)
                m.share_prefix(B)
                m.prefill_padded(body, lens, la)
                binding.op_greedy(la, na)

            def recompute():
                m.set_length(0, 0)
                m.prefill_padded(full, lens + P, lb)
                binding.op_greedy(lb, nb)

            ms_a = _timed(torch, shared, K, Wm)
            ms_b = _timed(torch, recompute, K, Wm)
            shared()
            recompute()
            torch.cuda.synchronize()
            agree = float((na == nb).float().mean().item())
            line.update({"batch": B, "prefix": P, "prompt_tokens": int(lens.sum()), "shared_ms": ms_a,
                         "recompute_ms": ms_b, "speedup": ms_b / ms_a, "first_token_agreement": agree,
                         "logits_rel_l2": float((la - lb).norm() / lb.norm())})
            assert m.get_error() == 0
            m.close()
        elif args.feature == "window":
            W = 4096
            cfg = dict(configs.QWEN3_8B, sliding_window=W, rolling_cache=1)
            V, L, Hkv, dh = cfg["vocab"], cfg["n_layers"], cfg["n_kv_heads"], cfg["head_dim"]
            seed = 7
            w = synth.make_weights(cfg, seed, device=dev)
            Bd, ctx, D = 16, 32768, 64
            m = binding.Model(cfg, w, max_batch=Bd, capacity=ctx + D + 8, max_tokens=128)
            k0, _ = m.kv_view(0)
            R = k0.shape[2]
            for layer in range(L):
                k, v = m.kv_view(layer)
                shape = (Bd, Hkv, R, dh)
                k.copy_(synth.make_kv_normal(shape, seed, layer, "k", device=dev))
                v.copy_(synth.make_kv_normal(shape, seed, layer, "v", device=dev))
            nxt = synth.make_ids(V, Bd, 1, seed, device=dev).reshape(Bd)
            logits = torch.empty(Bd, V, dtype=torch.float32, device=dev)
            m.set_length(ctx, Bd)

            def decode():
                m.decode_step(nxt, logits)
                binding.op_greedy(logits, nxt)

            dms = _timed(torch, decode, D - 3, 3)
            m.set_length(ctx, Bd)
            kern = _kernel_split(m, lambda: m.decode_step(nxt, logits), 8)
            att_bytes = 2.0 * Bd * Hkv * W * dh * 2
            att_ms = kern.get("attn_decode", 0) / L
            full_cache = 2.0 * L * Bd * Hkv * (ctx + D + 8) * dh * 2
            line.update({"window": W, "decode_batch": Bd, "context": ctx, "ring_slots": R,
                         "decode_ms_per_step": dms, "decode_kernels_ms": kern,
                         "attn_decode_gbs": att_bytes / (att_ms / 1e3) / 1e9 if att_ms else None,
                         "attn_decode_frac_of_hbm": att_bytes / (att_ms / 1e3) / 1e9 / peaks["hbm_gbs"] if att_ms else None,
                         "cache_gb": 2.0 * L * Bd * Hkv * R * dh * 2 / 1e9, "full_cache_gb": full_cache / 1e9})
            assert m.get_error() == 0
            m.close()
            # banded prefill of one long sequence over a full cache
            cfgb = dict(configs.QWEN3_8B, sliding_window=W, rolling_cache=0)
            T = 32768
            mb = binding.Model(cfgb, w, max_batch=1, capacity=T, max_tokens=T)
            ids = synth.make_ids(V, 1, T, seed, device=dev)
            lg = torch.empty(1, V, dtype=torch.float32, device=dev)

            def prefill():
                mb.set_length(0, 0)
                mb.prefill(ids, lg)

            pms = _timed(torch, prefill, max(1, K // 4), 3)
            kern = _kernel_split(mb, prefill, 1)
            pairs = W * (W + 1) / 2 + (T - W) * W
            att_flops = 4.0 * cfgb["n_q_heads"] * dh * pairs
            line.update({"banded_prefill_tokens": T, "banded_prefill_ms": pms,
                         "banded_prefill_tokens_per_s": T / (pms / 1e3), "banded_prefill_kernels_ms": kern,
                         "banded_attn_tflops": att_flops * L / (kern["attn_prefill"] / 1e3) / 1e12})
            assert mb.get_error() == 0
            mb.close()
        else:
            raise SystemExit(f"unknown feature {args.feature}")
    line["clocks"] = clk.summary()
    print(json.dumps(line), flush=True)



def _flat(w):
    for k, v in w.items():
        if isinstance(v, list):
            for t in v:
                if t is not None:
                    yield k, t
        elif v is not None:
            yield k, v


def main():
    from qwen3_decoder_transformer_gb300 import configs
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(configs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-steps", type=int, default=128, help="cap on timed decode steps")
    ap.add_argument("--op", default=None, help="time one kernel alone: attn_prefill, attn_decode, gemm_gateup, "
                                                "gemm_qkv, gemm_o, gemm_down, gemm_o_norm, qknorm_rope, rmsnorm, "
                                                "embed, greedy; or decode_step (whole decode steps)")
    ap.add_argument("--feature", default=None, choices=["padded", "prefix", "window"],
                    help="time a generation feature on its own workload instead of the step")
    ap.add_argument("--kv-split", type=int, default=0, help="--op attn_prefill: minimum tiles per KV chunk")
    ap.add_argument("--kv-chunks", type=int, default=1, help="--op attn_prefill: maximum KV chunks per query tile")
    ap.add_argument("--heads", type=int, default=0, help="--op attn_prefill: query heads per CTA (0 = automatic)")
    ap.add_argument("--len0", type=int, default=0, help="--op attn_prefill: cached tokens before the chunk")
    ap.add_argument("--rows", type=int, default=0,
                    help="row count for --op gemm_*/rmsnorm/embed (default B*T), batch for --op attn_decode, "
                         "greedy and decode_step")
    ap.add_argument("--layers", type=int, default=0,
                    help="--op decode_step: build only this many layers (small device footprint for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = configs.WORKLOADS[args.workload]
    if args.feature:
        run_feature(args)
    elif args.op:
        run_op(args, wl)
    elif args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
