"""Throughput of the attention forward on one GB300 (or N replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME]

One step is one fa_fwd call (the whole hot path) over one batch of the
workload's synthetic inputs, already resident in device memory. Rank 0 prints
one JSON line. With N > 1 (torchrun, one rank per GPU) every rank runs its
own replica of the workload (weak scaling; the path needs no collective), and
the timed region is bracketed by barriers; the max time over ranks is used.

--impl reference times the fp64 CPU oracle instead (bounded row samples of the
same workload per step) on the host cores, on rank 0 only.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from exact_attention_16_gb300 import metrics  # noqa: E402
from exact_attention_16_gb300.workloads import WORKLOADS, by_name, draw_inputs  # noqa: E402

DEFAULT_WORKLOAD = "causal_gqa8_b1_s16384"
L2_BYTES = 129 * 1000 * 1000
DATASHEET_BF16_TFLOPS = 2250.0   # GB300 dense BF16/FP16 tensor peak (nominal, without 2:4 sparsity)
METRIC = "attention fwd TFLOP/s (unmasked FLOPs) and % of GB300 dense BF16 tensor peak"
KERNEL_SOURCES = ["exact_attention_16_gb300/csrc/fa_fwd_kernel.cuh", "exact_attention_16_gb300/csrc/ptx_sm103.cuh",
                  "exact_attention_16_gb300/csrc/softmax_row.cuh"]
TRAFFIC_SUMMARY = "profiles/fa_fwd_kernel_traffic.md"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": d["bf16_tflops"], "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "source": "fallback"}


def exp_roofline(flop, D, avg_launch_ms):
    """The softmax's roof: one exp per unmasked (query, key) pair (FLOPs / 4D)
    per launch, against the probe-measured MUFU ex2 rate."""
    peak = ex2_peak_per_s()
    achieved = flop / (4.0 * D) / (avg_launch_ms * 1e-3)
    return {"bound": "mufu_ex2", "achieved": round(achieved / 1e9, 1),
            "peak": round(peak / 1e9, 1) if peak else None, "unit": "Gexp/s",
            "frac": round(achieved / peak, 4) if peak else None,
            "peak_source": "ex2 throughput probe on this GPU (libfa_probes.so)" if peak else "probe unavailable"}


def ex2_peak_per_s():
    """MUFU ex2 throughput of the current GPU, measured by the probe library
    (4 blocks per SM x 256 threads x 8 independent ex2 chains), or None."""
    import ctypes

    import torch

    path = os.path.join(ROOT, "exact_attention_16_gb300", "_lib", "libfa_probes.so")
    if not os.path.exists(path):
        return None
    lib = ctypes.CDLL(path)
    lib.fa_probe_ex2_rate.restype = ctypes.c_int
    lib.fa_probe_ex2_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p]
    rate = ctypes.c_double(0.0)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    rc = lib.fa_probe_ex2_rate(4 * sms, 2048, ctypes.byref(rate),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rate.value if rc == 0 else None


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source for this workload (else None)."""
    path = os.path.join(ROOT, TRAFFIC_SUMMARY)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha") != kernel_source_hash() or fields.get("workload") != workload:
        return None
    try:
        return int(float(fields["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.4)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                clk, cmax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            sm.append(clk)
            mx = cmax
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(value: float, dist, device) -> float:
    """Largest `value` over all ranks (the slowest rank's time); identity
    when `dist` is None. A control-plane reduction, not part of the step."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flop_per_step: int, steps: int, max_ms: float) -> float:
    """Aggregate throughput: every rank ran `steps` steps of `flop_per_step`
    (weak scaling); the job took as long as the slowest rank."""
    return world * flop_per_step * steps / (max_ms * 1e-3) / 1e12


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_ours(args, w):
    import torch

    from exact_attention_16_gb300 import api

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = dist_mod
    dev = torch.device("cuda", local)
    q, k, v = draw_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.fa_fwd(qd, kd, vd, scale=w.scale, causal=w.causal, out=out, lse=lse)

    for _ in range(args.warmup):
        step()
    if api.fa_status() != 0:
        raise RuntimeError("device status not OK after warm-up")

    flop = metrics.flops(w.B, w.Sq, w.Sk, w.Hq, w.D, w.causal)
    in_bytes = sum(x.numel() * x.element_size() for x in (q, k, v))
    # Inputs larger than L2 are timed back to back. Smaller ones get an L2
    # flush (a 256 MiB write) before every launch, and the step time is then
    # the sum of the per-launch event intervals, which exclude the flush.
    flush = None if in_bytes > L2_BYTES else torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    l2_note = (f"inputs larger than L2 (q+k+v = {in_bytes >> 20} MiB > 129 MB); no flush" if flush is None
               else f"inputs ({in_bytes >> 20} MiB) smaller than L2: 256 MiB L2 flush before each launch, "
                    "flush excluded from the per-launch event timing")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    if api.fa_status() != 0:
        raise RuntimeError("device status not OK after the timed region")
    launch_ms = [starts[i].elapsed_time(ends[i]) for i in range(args.steps)]
    total_ms = starts[0].elapsed_time(ends[-1]) if flush is None else sum(launch_ms)
    total_ms = max_over_ranks(total_ms, dist, dev)

    # end to end through the public call for host tensors (fa_fwd_host) with
    # pinned host buffers: every step copies q, k, v in, runs the kernels and
    # copies O and LSE out, pipelined per chunk inside the call
    hq_, hk_, hv_ = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    ws = torch.empty(api.fa_fwd_host_workspace_size(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D), dtype=torch.uint8,
                     device=dev)
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        api.fa_fwd_host(hq_, hk_, hv_, scale=w.scale, causal=w.causal, out=ho, lse=hl, workspace=ws,
                        synchronize=False)

    e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)
    h2d = in_bytes
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()

    peaks = measured_peaks()
    avg_launch_ms = sum(launch_ms) / len(launch_ms)
    achieved = flop / (avg_launch_ms * 1e-3) / 1e12
    value = whole_job_tflops(world, flop, args.steps, total_ms)
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded PCG64 normal draws rounded to the dtype)",
        "config": {
            "workload": w.name, "B": w.B, "Sq": w.Sq, "Sk": w.Sk, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
            "causal": w.causal, "scale": w.scale, "flops_per_step": flop,
            "l2": l2_note,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "pct_of_peak": round(100.0 * (value / world) / peaks["bf16_tflops"], 2),
        "pct_of_peak_source": peaks["source"] + " bf16 burst (cuBLAS)",
        "pct_of_datasheet_peak": round(100.0 * (value / world) / DATASHEET_BF16_TFLOPS, 2),
        "roofline": {
            "bound": "tensor",
            "achieved": round(achieved, 2),
            "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": round(achieved / peaks["bf16_tflops"], 4),
            "peak_source": peaks["source"] + " bf16 burst",
            "traffic": recorded_traffic(w.name),
            "algorithmic_bytes": metrics.algorithmic_bytes(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D),
            "kernel": "fa_fwd_kernel" if w.D <= 128 else "fa_decode_kernel",
            "avg_launch_ms": round(avg_launch_ms, 4),
        },
        "exp_roofline": exp_roofline(flop, w.D, avg_launch_ms),
        "e2e": {
            "value": round(whole_job_tflops(world, flop, e2e_steps, e2e_s * 1e3), 2),
            "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "call": "fa_fwd_host (pinned host tensors; copies pipelined with the kernels per chunk)",
        },
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, q, k, v, budget_s=args.cpu_budget)
    if dist:
        dist.destroy_process_group()
    return rank, result


def run_merge(args, w):
    """Merge of `args.parts` partial (O, LSE) states shaped like the
    workload's output (the exchange step of a context-parallel run):
    HBM-bound, reported in GB/s of algorithmic bytes."""
    import torch

    from exact_attention_16_gb300 import api

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    n = args.parts
    g = torch.Generator(device=dev).manual_seed(w.seed)
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[w.dtype]
    o_parts = torch.randn((n, w.B, w.Sq, w.Hq, w.D), generator=g, device=dev).to(dt)
    lse_parts = torch.randn((n, w.B, w.Hq, w.Sq), generator=g, device=dev) * 3
    out = torch.empty((w.B, w.Sq, w.Hq, w.D), dtype=dt, device=dev)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    rows = w.B * w.Sq * w.Hq
    nbytes = n * rows * w.D * 2 + n * rows * 4 + rows * w.D * 2 + rows * 4

    def step():
        api.fa_merge(o_parts, lse_parts, out=out, lse=lse)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stream = torch.cuda.current_stream(dev)
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    launch_ms = [starts[i].elapsed_time(ends[i]) for i in range(args.steps)]
    total_ms = starts[0].elapsed_time(ends[-1])
    peaks = measured_peaks()
    avg = sum(launch_ms) / len(launch_ms)
    value = nbytes * args.steps / (total_ms * 1e-3) / 1e9
    return rank, {
        "metric": "attention partial-state merge GB/s (algorithmic bytes)",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded torch normal draws)",
        "config": {"workload": f"merge {n} parts shaped like {w.name}", "parts": n, "B": w.B, "Sq": w.Sq,
                   "Hq": w.Hq, "D": w.D, "bytes_per_step": nbytes,
                   "l2": f"inputs {nbytes >> 20} MiB > 129 MB L2; no flush"},
        "roofline": {"bound": "hbm", "achieved": round(nbytes / (avg * 1e-3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(nbytes / (avg * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"] + " copy bandwidth", "traffic": None, "kernel": "merge_kernel",
                     "avg_launch_ms": round(avg, 4)},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }


def run_decode(args, w):
    """Split-KV decode: one query position per sequence against the
    workload's keys, batch `args.decode_batch`. HBM-bound (every K/V byte is
    read once per step), reported in GB/s of algorithmic bytes."""
    import torch

    from exact_attention_16_gb300 import api
    from exact_attention_16_gb300.workloads import Workload

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wd = Workload(f"decode_{w.name}", args.decode_batch, 1, w.Sk, w.Hq, w.Hkv, w.D, w.dtype, True, w.sigma_qk,
                  w.sigma_v, w.seed)
    q, k, v = (t.to(dev) for t in draw_inputs(wd))
    out = torch.empty_like(q)
    lse = torch.empty((wd.B, wd.Hq, 1), dtype=torch.float32, device=dev)
    need = api.fa_decode_workspace_size(wd.B, 1, wd.Sk, wd.Hq, wd.Hkv, wd.D, 0)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    nbytes = metrics.algorithmic_bytes(wd.B, 1, wd.Sk, wd.Hq, wd.Hkv, wd.D)

    def step():
        api.fa_fwd_decode(q, k, v, scale=wd.scale, causal=True, workspace=ws, out=out, lse=lse)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if args.graph:
        # One step captured in a CUDA graph and replayed: at a few sequences a
        # step's GPU time is below the host cost of one eager call through
        # the binding, which the eager loop would otherwise measure.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        step = graph.replay
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    if api.fa_status() != 0:
        raise RuntimeError("device status not OK")
    launch_ms = [starts[i].elapsed_time(ends[i]) for i in range(args.steps)]
    total_ms = starts[0].elapsed_time(ends[-1])
    peaks = measured_peaks()
    avg = sum(launch_ms) / len(launch_ms)
    value = nbytes * args.steps / (total_ms * 1e-3) / 1e9
    return rank, {
        "metric": "decode attention GB/s (algorithmic bytes: Q, K, V read once, O and LSE written once)",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wd.dtype, "data": "synthetic (seeded PCG64 normal draws rounded to the dtype)",
        "config": {"workload": wd.name, "B": wd.B, "Sq": 1, "Sk": wd.Sk, "Hq": wd.Hq, "Hkv": wd.Hkv, "D": wd.D,
                   "bytes_per_step": nbytes, "workspace_bytes": need,
                   "launch": "CUDA graph replay per step" if args.graph else "eager call per step",
                   "l2": f"K+V {nbytes >> 20} MiB" + (" > 129 MB L2; no flush" if nbytes > L2_BYTES else
                                                       " (smaller than L2: hot-L2 figure)")},
        "roofline": {"bound": "hbm", "achieved": round(nbytes / (avg * 1e-3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(nbytes / (avg * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"] + " copy bandwidth", "traffic": None,
                     "kernel": "fa_decode_kernel + merge_kernel", "avg_launch_ms": round(avg, 4)},
        "gpu_launches": 2 * args.steps if need > 0 else args.steps,
        "clocks": clocks.summary(),
    }


def run_splitkv(args, w):
    """The workload as given through the split-KV path (fa_fwd_decode), which
    serves small prefill problems that leave fa_fwd's persistent grid
    partly idle; same TFLOP/s metric as the default leg."""
    import torch

    from exact_attention_16_gb300 import api

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v = (t.to(dev) for t in draw_inputs(w))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    need = api.fa_decode_workspace_size(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D, 0)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    flop = metrics.flops(w.B, w.Sq, w.Sk, w.Hq, w.D, w.causal)
    in_bytes = sum(x.numel() * x.element_size() for x in (q, k, v))
    flush = None if in_bytes > L2_BYTES else torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        api.fa_fwd_decode(q, k, v, scale=w.scale, causal=w.causal, workspace=ws, out=out, lse=lse)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    if api.fa_status() != 0:
        raise RuntimeError("device status not OK")
    launch_ms = [starts[i].elapsed_time(ends[i]) for i in range(args.steps)]
    total_ms = starts[0].elapsed_time(ends[-1]) if flush is None else sum(launch_ms)
    peaks = measured_peaks()
    value = whole_job_tflops(1, flop, args.steps, total_ms)
    return rank, {
        "metric": METRIC + " (split-KV path)", "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded PCG64 normal draws rounded to the dtype)",
        "config": {"workload": w.name, "path": "fa_fwd_decode", "workspace_bytes": need,
                   "l2": "no flush (inputs > L2)" if flush is None else
                         "256 MiB L2 flush before each launch, excluded from the event timing"},
        "pct_of_peak": round(100.0 * value / peaks["bf16_tflops"], 2),
        "gpu_launches": (2 if need > 0 else 1) * args.steps,
        "clocks": clocks.summary(),
    }


def oracle_sample(w, q32, k32, v32, rows_per_head: int, n_heads: int):
    """Time the oracle on the last `rows_per_head` rows of the first heads;
    returns (seconds, flops done)."""
    import oracle

    flop = 0
    t0 = time.perf_counter()
    for idx in range(n_heads):
        b, hq = divmod(idx % (w.B * w.Hq), w.Hq)
        rows = np.arange(max(0, w.Sq - rows_per_head), w.Sq)
        oracle.attention_rows(q32, k32, v32, w.scale, w.causal, b, hq, rows)
        flop += 4 * w.D * sum(metrics.visible_keys(int(i), w.Sq, w.Sk, w.causal) for i in rows)
    return time.perf_counter() - t0, flop


def cpu_baseline(w, q, k, v, budget_s: float):
    q32, k32, v32 = q.float().numpy(), k.float().numpy(), v.float().numpy()
    rows = min(w.Sq, 256)
    heads = 1
    secs, flop = oracle_sample(w, q32, k32, v32, rows, heads)
    # grow the sample (more heads, then more rows per head) until one pass
    # takes at least two thirds of `budget_s`
    while secs < budget_s * 0.66 and (heads < w.B * w.Hq or rows < w.Sq):
        if heads < w.B * w.Hq:
            heads = min(w.B * w.Hq, heads * 2)
        else:
            rows = min(w.Sq, rows * 2)
        secs, flop = oracle_sample(w, q32, k32, v32, rows, heads)
    return {
        "value": round(flop / secs / 1e12, 6),
        "unit": "TFLOP/s",
        "cores": int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1)),
        "kind": "oracle",
        "sample": f"fp64 NumPy two-pass oracle on the last {rows} query rows of {heads} (batch, head) pairs "
                  f"of {w.name} ({secs:.1f} s; BLAS threads = cores, elementwise NumPy single-threaded)",
    }


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return rank, None
    q, k, v = draw_inputs(w)
    q32, k32, v32 = q.float().numpy(), k.float().numpy(), v.float().numpy()
    # size one step so that warm-up + timed steps take about two minutes
    per_step_s = max(0.05, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    rows = 16
    secs, _ = oracle_sample(w, q32, k32, v32, rows, 1)
    while secs < per_step_s * 0.5 and rows < w.Sq:
        rows = min(w.Sq, rows * 2)
        secs, _ = oracle_sample(w, q32, k32, v32, rows, 1)
    for _ in range(args.warmup):
        oracle_sample(w, q32, k32, v32, rows, 1)
    t_total, f_total = 0.0, 0
    for _ in range(args.steps):
        s, f = oracle_sample(w, q32, k32, v32, rows, 1)
        t_total += s
        f_total += f
    value = f_total / t_total / 1e12
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    sample = f"fp64 NumPy two-pass oracle, last {rows} query rows of (b=0, h=0) of {w.name} per step"
    return rank, {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_total / max(1, args.steps), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded PCG64 normal draws rounded to the dtype)",
        "config": {"workload": w.name, "B": w.B, "Sq": w.Sq, "Sk": w.Sk, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "causal": w.causal},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["fwd", "merge", "decode", "splitkv"], default="fwd",
                    help="fwd: the attention forward (default); merge: partial-state merge; decode: split-KV "
                         "decode; splitkv: the workload through the split-KV path")
    ap.add_argument("--decode-batch", type=int, default=16, help="sequences per step for --op decode")
    ap.add_argument("--graph", action="store_true", help="--op decode: replay each step from a CUDA graph")
    ap.add_argument("--parts", type=int, default=4, help="partial states for --op merge")
    ap.add_argument("--head-dim", type=int, default=0, help="override the workload's head dimension (64/128/256)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=[x.name for x in WORKLOADS])
    ap.add_argument("--cpu-budget", type=float, default=18.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = by_name(args.workload)
    if args.head_dim:
        w = w.with_sizes(D=args.head_dim, name=f"{w.name}_d{args.head_dim}")
    if args.impl == "reference":
        rank, res = run_reference(args, w)
    elif args.op == "merge":
        rank, res = run_merge(args, w)
    elif args.op == "decode":
        rank, res = run_decode(args, w)
    elif args.op == "splitkv":
        rank, res = run_splitkv(args, w)
    else:
        rank, res = run_ours(args, w)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
