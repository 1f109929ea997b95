"""Benchmark of the FLARE++ mixer forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one full mixer forward (synthesis, gate, encode, decode) over one
batch of the chosen synthetic workload (default: the industrial-aero-shaped
workload, B=1 H=8 N=1048576 M=512 D=32, bf16 -- the largest of the paper's
workloads that fits one GPU). Prints one JSON line.

Device timing: W warm-up steps, then exactly K steps, each bracketed by CUDA
events on the launching stream, with a 512 MB L2 flush before every step
(outside the events). Under torchrun each rank runs its own replica of the
workload (weak scaling, no collective on the data path); a barrier and
torch.cuda.synchronize() bracket the timed region and the slowest rank's time
counts. ``e2e`` times the same call with the inputs copied from pinned host
memory and the output copied back inside the timed region.

``--impl reference`` times the CPU fp64 oracle (the only reference this path
has) on a bounded sample of the same workload, on the host cores.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rank_latent_routing_gb300 import workloads  # noqa: E402

METRIC = "FLARE++ mixer fwd tokens/s and TFLOP/s (% of bf16 roofline) at 1 GB300"
UNIT = "tokens/s"

# Fallback denominators (used only if MEASURED_PEAKS.json is missing).
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}
# exp2 results per clock per SM on the special-function unit: 32 on GB300
# (measured by python -m rank_latent_routing_gb300.micro, record in
# profiles/issue_rates_gb300.md; twice B200's 16)
MUFU_EX2_PER_CLK_PER_SM = 32


def sm_count(device=None) -> int:
    """Streaming multiprocessors of the device, read at run time."""
    import torch
    d = torch.cuda.current_device() if device is None else device
    return int(torch.cuda.get_device_properties(d).multi_processor_count)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for ts, line in self.lines:
            if ts < t0 - 0.15 or ts > t1 + 0.15:
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- our path
# inputs each mixer variant reads (the library refuses others)
VARIANT_INPUTS = {
    "flarepp": ("K", "V", "Ks_raw", "Qseed", "Qf", "gate"),
    "unshared": ("K", "V", "Ks_raw", "Vs", "Qseed", "Qf", "gate"),
    "simplified": ("K", "V", "Ks_raw", "Vs", "Qseed"),
    "flare": ("Qlat", "K", "V"),
}


def upload(wl, torch, device, variant="flarepp"):
    names = VARIANT_INPUTS[variant]
    ex = workloads.variant_inputs(wl) if ("Vs" in names or "Qlat" in names) else {}
    out = {}
    for k in names:
        if k == "gate":
            out[k] = torch.from_numpy(wl.gate)
        elif wl.dtype == "bf16":
            bits = ex[k + "_bits"] if k in ex else wl.bits[k]
            out[k] = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(ex[k] if k in ex else getattr(wl, k)))
    dev = {k: v.to(device) for k, v in out.items()}
    host = {k: v.pin_memory() for k, v in out.items()}
    return dev, host


def stage_costs(s: workloads.Shape, es: int, variant: str = "flarepp"):
    """Algorithmic work of each pass per call: bytes moved, flops, exps.

    Per (token, head): synthesis reads Ks_raw (D elements; 2D with separate
    values Vs; nothing for FLARE, which has no synthesis); encode reads K and
    V (2D); decode reads K and writes Y (2D). Each pass scores N x M and
    multiplies by a D-wide value: 4*M*D flops and M exponentials per token.
    Latent-sized traffic (Qseed, Qf, Q, Z, partials) is below 1% and not counted.
    """
    th = s.B * s.H * s.N
    per_pass_flops = 4.0 * th * s.M * s.D
    per_pass_exps = float(th) * s.M
    synth = {"flarepp": 1, "unshared": 2, "simplified": 2, "flare": 0}[variant]
    return {
        "synthesis": {"bytes": synth * th * s.D * es, "flops": per_pass_flops * (synth > 0),
                      "exps": per_pass_exps * (synth > 0)},
        "encode": {"bytes": 2 * th * s.D * es, "flops": per_pass_flops, "exps": per_pass_exps},
        "decode": {"bytes": 2 * th * s.D * es, "flops": per_pass_flops, "exps": per_pass_exps},
    }


def roofline(costs, stage_ms, peaks, peak_kind, clock_mhz, sms):
    """The dominant pass against the resource that bounds it.

    Ideal times: bytes / HBM peak, flops / bf16 tensor peak, exps / MUFU exp2
    peak (32 per clock per SM x the device's SMs x the max SM clock). The
    bound is the resource with the longest ideal time; frac = that ideal time
    / measured.
    """
    name = max(stage_ms, key=lambda k: stage_ms[k])
    c = costs[name]
    t = stage_ms[name] * 1e-3
    hbm = peaks["hbm_gbs"] * 1e9
    tensor = peaks["bf16_tflops_sustained"] * 1e12
    exp_peak = MUFU_EX2_PER_CLK_PER_SM * sms * peaks.get("sm_max_mhz", 2070.0) * 1e6
    ideal = {"hbm": c["bytes"] / hbm, "tensor": c["flops"] / tensor, "alu": c["exps"] / exp_peak}
    bound = max(ideal, key=lambda k: ideal[k])
    if bound == "hbm":
        ach, pk, unit = c["bytes"] / t / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "tensor":
        ach, pk, unit = c["flops"] / t / 1e12, peaks["bf16_tflops_sustained"], "TFLOP/s"
    else:
        ach, pk, unit = c["exps"] / t / 1e9, exp_peak / 1e9, "Gexp/s"
    return {"bound": bound, "kernel": name, "achieved": round(ach, 3), "peak": round(pk, 3),
            "unit": unit, "frac": round(ach / pk, 4), "traffic": None,
            "peak_source": peak_kind + (f" (MUFU exp2 peak: measured 32/clk/SM x {sms} SMs x max "
                                        "SM clock)" if bound == "alu" else ""),
            "ideal_us": {k: round(v * 1e6, 3) for k, v in ideal.items()},
            "stage_ms": {k: round(v, 5) for k, v in stage_ms.items()},
            "hbm_frac": round(c["bytes"] / t / hbm, 4),
            "tensor_frac": round(c["flops"] / t / tensor, 4)}


def max_over_ranks(values, world, device):
    """Element-wise maximum of per-rank timings (the slowest rank counts)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


TC_SOURCE = os.path.join(ROOT, "rank_latent_routing_gb300", "csrc", "tc.cu")
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "roofline_traffic.md")


def measured_traffic(workload: str, kernel: str, src: str = TC_SOURCE, prof: str = TRAFFIC_RECORD):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary (profiles/roofline_traffic.md), or None when it was measured on a
    different revision of the tensor-core kernels (source hash mismatch)."""
    import hashlib
    if not (os.path.exists(src) and os.path.exists(prof)):
        return None
    with open(src, "rb") as f:
        sha = hashlib.sha1(f.read()).hexdigest()[:12]
    with open(prof) as f:
        for line in f:
            if not line.startswith("traffic:"):
                continue
            fields = dict(kv.split("=", 1) for kv in line[len("traffic:"):].split())
            if (fields.get("workload") == workload and fields.get("kernel") == kernel
                    and fields.get("source_sha1") == sha):
                return int(fields["bytes_per_launch"])
    return None


def workload_string(name: str, variant: str = "flarepp", tokens: int = 0) -> str:
    """The ``config.workload`` string, the same for both arms of the bench
    (``tokens`` > 0: the workload cut to that many tokens per head, a
    profiling case, named as such)."""
    s, dtype = workloads.CONFIGS[name][0], workloads.CONFIGS[name][1]
    n = tokens if tokens > 0 else s.N
    return (f"{name}{' cut to N=' + str(n) if tokens > 0 else ''}: B={s.B} H={s.H} N={n} M={s.M} D={s.D} {dtype}"
            + ("" if variant == "flarepp" else f", {variant} mixer"))


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from rank_latent_routing_gb300 import flarepp

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = workloads.config(args.workload, **({"N": args.tokens} if args.tokens > 0 else {}))
    s = wl.shape
    dev, host = upload(wl, torch, device, args.variant)
    tdtype = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    out = torch.empty(s.B, s.H, s.N, s.D, dtype=tdtype, device=device)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step():
        if args.variant == "flarepp":
            flarepp.forward(dev["K"], dev["V"], dev["Ks_raw"], dev["Qseed"], dev["Qf"],
                            dev["gate"], out=out)
        elif args.variant == "flare":
            flarepp.flare_forward(dev["Qlat"], dev["K"], dev["V"], out=out)
        else:
            flarepp.forward_variant(args.variant, dev["K"], dev["V"], dev["Ks_raw"], dev["Vs"],
                                    dev["Qseed"], dev.get("Qf"), dev.get("gate"), out=out)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if flarepp.sync_status() != 0:
        raise RuntimeError("device error during warm-up")

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    timer = flarepp.StageTimer()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stage_sum = [0.0, 0.0, 0.0]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        if i % 8 == 0:
            with timer:
                step()
            ends[i].record(stream)
            for j, v in enumerate(timer.elapsed_ms()):
                stage_sum[j] += v
        else:
            step()
            ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t1 = time.time()
    clk = clocks.stop(t0, t1)
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(ms)
    if flarepp.sync_status() != 0:
        raise RuntimeError("device error in timed region")
    n_stage = len(range(0, args.steps, 8))
    stage_ms = {k: v / n_stage for k, v in zip(("synthesis", "encode", "decode"), stage_sum)}

    # end to end through the public call: pinned host inputs in, result out
    e2e_steps = max(5, min(args.steps, 50))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = hout.numel() * hout.element_size()
    for _ in range(2):
        for k in dev:
            dev[k].copy_(host[k], non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        for k in dev:
            dev[k].copy_(host[k], non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    t_max, e2e_max = max_over_ranks([total_ms, e2e_ms], world, device)
    if rank != 0:
        return None

    peaks, kind = load_peaks()
    tokens = s.tokens * world
    ms_step = t_max / args.steps
    value = tokens / (ms_step * 1e-3)
    passes = 2 if args.variant == "flare" else 3
    tflops = s.flops * passes / 3 * world / (ms_step * 1e-3) / 1e12
    costs = stage_costs(s, 2 if wl.dtype == "bf16" else 4, args.variant)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "ms_median": round(float(np.median(ms)), 5), "ms_min": round(float(min(ms)), 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic (seeded, shapes of the paper's workloads)",
        "config": {"workload": workload_string(args.workload, args.variant, args.tokens),
                   "global_batch": s.B * world, "seq_len": s.N, "latents": s.M, "head_dim": s.D,
                   "heads": s.H, "parallelism": f"replicas x{world}" if world > 1 else "single",
                   "l2": "512 MB flush before every timed step"},
        "tflops": round(tflops, 3),
        "tensor_roofline_frac": round(tflops / peaks["bf16_tflops_sustained"], 4),
        "roofline": roofline(costs, stage_ms, peaks, kind, clk.get("sm_mhz"), sm_count(device)),
        "clocks": clk,
        "e2e": {"value": round(tokens / (e2e_max * 1e-3), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_max, 4)},
        "gpu_launches": passes * args.steps,
        "impl": "ours",
    }
    rl = line["roofline"]
    rl["traffic"] = (measured_traffic(args.workload, rl["kernel"])
                     if args.variant == "flarepp" and args.tokens <= 0 else None)
    return line


def run_project(args, rank, world, local_rank):
    """The fused token projections (K = N_a(X W_K), V = X W_V, raw synthesis
    keys) on the workload's B, H, N, D: X [B, N, H D] in, three [B, H, N, D]
    out. HBM-bound at these widths; reported against the measured copy peak."""
    import torch
    from rank_latent_routing_gb300 import flarepp

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    s = workloads.CONFIGS[args.workload][0]
    pr = workloads.projection_inputs(s.B, s.H, s.N, s.D, dtype="bf16", seed=3)
    C = s.H * s.D
    host = {"X": torch.from_numpy(np.ascontiguousarray(pr.bits["X"]).view(np.int16)).view(torch.bfloat16),
            "W": torch.from_numpy(np.ascontiguousarray(pr.bits["W"]).view(np.int16)).view(torch.bfloat16),
            "bias": torch.from_numpy(pr.bias), "scales": torch.from_numpy(pr.scales)}
    dev = {k: v.to(device) for k, v in host.items()}
    host = {k: v.pin_memory() for k, v in host.items()}
    outs = [torch.empty(s.B, s.H, s.N, s.D, dtype=torch.bfloat16, device=device) for _ in range(3)]
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step():
        flarepp.project(dev["X"], dev["W"], s.H, pr.norms, bias=dev["bias"], scales=dev["scales"],
                        outs=outs)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if flarepp.sync_status() != 0:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    clk = clocks.stop(t0, t1)
    if flarepp.sync_status() != 0:
        raise RuntimeError("device error in timed region")
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps

    # end to end: X from pinned host memory in, the three outputs back
    hout = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    e2e_steps = max(5, min(args.steps, 20))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        dev["X"].copy_(host["X"], non_blocking=True)
        step()
        for h, o in zip(hout, outs):
            h.copy_(o, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    t_max, e2e_max = max_over_ranks([ms, e2e_ms], world, device)
    if rank != 0:
        return None
    peaks, kind = load_peaks()
    tokens = s.B * s.N * world
    nbytes = s.B * s.N * C * 2 * 4 + 3 * C * C * 2  # X in, three outputs out, the weights once
    flops = 2.0 * s.B * s.N * C * 3 * C
    t = t_max * 1e-3
    ach = nbytes / t / 1e9
    return {
        "metric": "FLARE++ token projections (K, V, synthesis keys) tokens/s", "value": round(tokens / t, 1),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_max, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, near-identity weights)",
        "config": {"workload": f"projection of {args.workload}: B={s.B} N={s.N} C={C} (H={s.H} D={s.D}) "
                               "-> K (N_a), V, raw synthesis keys",
                   "l2": "512 MB flush before every timed step"},
        "roofline": {"bound": "hbm", "kernel": "proj_kernel", "achieved": round(ach, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                     "traffic": None, "peak_source": kind,
                     "tensor_frac": round(flops / t / 1e12 / peaks["bf16_tflops_sustained"], 4)},
        "clocks": clk,
        "e2e": {"value": round(tokens / (e2e_max * 1e-3), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(host["X"].numel() * 2),
                "d2h_bytes_per_step": int(sum(h.numel() * 2 for h in hout)),
                "ms_per_step": round(e2e_max, 4)},
        "gpu_launches": args.steps,
        "impl": "ours",
    }


FP32_FMA_PER_CLK_PER_SM = 128  # CUDA-core fp32 FMA lanes per SM per clock


def run_backward(args, rank, world, local_rank):
    """The mixer's backward pass (all input gradients for a random output
    cotangent) on the workload. It runs on the CUDA cores in fp32, so it is
    reported against the fp32 FMA peak (128 FMA lanes per SM per clock x SMs x
    the max SM clock) with 24 B H N M D algorithmic flops: each of the three
    attention calls costs four N x M x D products backward (scores, dP, and
    the two gradient products), twice the forward's two."""
    import torch
    from rank_latent_routing_gb300 import flarepp

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = workloads.config(args.workload)
    s = wl.shape
    dev, host = upload(wl, torch, device)
    ct = workloads.cotangent(wl)
    if wl.dtype == "bf16":
        dy = torch.from_numpy(np.ascontiguousarray(ct["dY_bits"]).view(np.int16)).view(torch.bfloat16).to(device)
    else:
        dy = torch.from_numpy(ct["dY"]).to(device)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step():
        return flarepp.backward(dev["K"], dev["V"], dev["Ks_raw"], dev["Qseed"], dev["Qf"], dev["gate"], dy)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if flarepp.sync_status() != 0:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    clk = clocks.stop(t0, t1)
    if flarepp.sync_status() != 0:
        raise RuntimeError("device error in timed region")
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    t_max = max_over_ranks([ms], world, device)[0]
    if rank != 0:
        return None
    peaks, kind = load_peaks()
    tokens = s.tokens * world
    t = t_max * 1e-3
    flops = 24.0 * s.B * s.H * s.N * s.M * s.D
    sms = sm_count(device)
    peak_tf = FP32_FMA_PER_CLK_PER_SM * 2 * sms * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    ach = flops / t / 1e12
    return {
        "metric": "FLARE++ mixer backward tokens/s", "value": round(tokens / t, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, shapes of the paper's workloads)",
        "config": {"workload": f"backward of {wl.name}: B={s.B} H={s.H} N={s.N} M={s.M} D={s.D} "
                               f"{wl.dtype} inputs, fp32 gradients",
                   "l2": "512 MB flush before every timed step"},
        "roofline": {"bound": "alu", "kernel": "backward passes (CUDA cores)", "achieved": round(ach, 3),
                     "peak": round(peak_tf, 3), "unit": "TFLOP/s", "frac": round(ach / peak_tf, 4),
                     "traffic": None,
                     "peak_source": f"fp32 FMA: 128 lanes/clk/SM x 2 flops x {sms} SMs x max SM clock"},
        "clocks": clk,
        "gpu_launches": 12 * args.steps,
        "impl": "ours",
    }


# ------------------------------------------------------------ CPU oracle
def _pool_init():
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"


_HEADS = {}


def _oracle_job(job):
    """One (batch, head) problem of the oracle on the first n_tok tokens;
    returns its wall time. The head's inputs are drawn once per process."""
    import oracle
    from rank_latent_routing_gb300 import workloads as w
    name, variant, b, h, n_tok = job
    key = (name, b, h)
    if key not in _HEADS:
        _HEADS[key] = w.make_head(name, b, h)
        if variant != "flarepp":
            _HEADS[key].update(w.make_variant_head(name, b, h))
    x = _HEADS[key]
    K, V = x["K"][:n_tok], x["V"][:n_tok]
    t0 = time.perf_counter()
    if variant == "flarepp":
        oracle.forward_head(K, V, x["Ks_raw"][:n_tok], x["Qseed"], x["Qf"], x["gate"])
    elif variant == "flare":
        oracle.flare_forward_head(x["Qlat"], K, V)
    else:
        args = (K[None, None], V[None, None], x["Ks_raw"][:n_tok][None, None],
                x["Vs"][:n_tok][None, None], x["Qseed"][None])
        if variant == "unshared":
            oracle.forward_unshared(*args, x["Qf"][None], np.array([x["gate"]]))
        else:
            oracle.forward_simplified(*args)
    return time.perf_counter() - t0


class OraclePool:
    """``cores`` spawned processes with one BLAS thread each; each runs whole
    (batch, head) problems of the workload through the unmodified oracle."""

    def __init__(self, name, cores, variant="flarepp"):
        import multiprocessing as mp
        self.name, self.cores, self.variant = name, cores, variant
        self.shape = workloads.CONFIGS[name][0]
        s = self.shape
        # each process draws its own heads; keep to `cores` distinct heads
        self.heads = [(i // s.H % s.B, i % s.H) for i in range(min(cores, s.B * s.H))]
        _pool_init()
        self.pool = mp.get_context("spawn").Pool(cores, initializer=_pool_init)
        self.round(min(s.N, 256))  # draw inputs, import modules

    def round(self, n_tok):
        jobs = [(self.name, self.variant, *self.heads[i % len(self.heads)], n_tok)
                for i in range(self.cores)]
        t0 = time.perf_counter()
        self.pool.map(_oracle_job, jobs, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def sample_tokens(pool, seconds: float) -> int:
    """Tokens per (batch, head) problem such that one round of the pool (one
    problem per process) takes about ``seconds``: whole problems where they
    are that quick, else the first n tokens of each (at least 128)."""
    s = pool.shape
    probe = min(s.N, 2048)
    t_probe = pool.round(probe)
    if t_probe * s.N / probe <= seconds:
        return s.N
    return max(128, min(s.N, int(probe * seconds / max(t_probe, 1e-9))))


def cpu_baseline(args):
    """The oracle's tokens/s on the host cores, on about ``--cpu-seconds`` of
    (batch, head) problems of the benchmark workload (each on its first n
    tokens where whole problems would take longer than a third of that)."""
    cores = os.cpu_count() or 1
    pool = OraclePool(args.workload, cores, args.variant)
    s = pool.shape
    n_tok = sample_tokens(pool, args.cpu_seconds / 3)
    done, el = 0, 0.0
    while el < args.cpu_seconds:
        el += pool.round(n_tok)
        done += cores
    pool.close()
    rate = done * n_tok / s.H / el
    return {"value": round(rate, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done} (batch, head) {args.variant} problems of {args.workload} on the first "
                      f"{n_tok} of N={s.N} tokens each, in {el:.1f} s on {cores} processes x 1 BLAS "
                      "thread; tokens/s = problems x tokens / H / wall time"}


def run_reference(args, rank, world):
    """Reference arm: the CPU fp64 oracle, one bounded sample per step."""
    if rank != 0:
        return None
    cores = os.cpu_count() or 1
    pool = OraclePool(args.workload, cores, args.variant)
    s = pool.shape
    budget = 120.0  # seconds for all warm-up and timed steps together
    per_step = max(0.05, budget / max(1, args.steps + args.warmup))
    n_tok = sample_tokens(pool, per_step)
    times = []
    for i in range(args.warmup + args.steps):
        t = pool.round(n_tok)
        if i >= args.warmup:
            times.append(t)
    pool.close()
    ms = 1e3 * sum(times) / len(times)
    value = cores * n_tok / s.H / (ms * 1e-3)
    return {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, shapes of the paper's workloads)",
            "config": {"workload": workload_string(args.workload, args.variant),
                       "parallelism": "host cores"},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": f"each step: {cores} (batch, head) problems on the first "
                                       f"{n_tok} of N={s.N} tokens, one process and one BLAS "
                                       "thread per core"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="aero", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--op", default="mixer", choices=["mixer", "project", "backward"],
                    help="what to time: the mixer forward, the fused token projections, or the "
                         "mixer's backward pass")
    ap.add_argument("--variant", default="flarepp", choices=sorted(VARIANT_INPUTS),
                    help="mixer: FLARE++ (default), separate synthesis values, simplified "
                         "FLARE++, or FLARE")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: cut the workload to this many tokens per head (mixer op)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run = {"mixer": run_ours, "project": run_project, "backward": run_backward}[args.op]
        line = run(args, rank, world, local_rank)
    finally:
        if world > 1:
            dist.destroy_process_group()
    if line is None:
        return
    if world == 1 and not args.no_cpu_baseline and args.op == "mixer":
        line["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
