#!/usr/bin/env python3
"""Benchmark of the GB300 MoE expert layer: tokens/s per layer vs prefill quantum.

One step = one moe_layer_forward over one serving step's token batch (router, top-k, grouping,
grouped gate/up + SwiGLU, down, combine, shared expert), inputs resident in HBM.

Default workload: the mixed prefill+decode step of the Qwen-A3B-like layer (d_model 2048,
256 experts, top-8, d_ff 512, one shared expert d_ff 512, bf16 weights) at prefill quantum
2048, i.e. T = 2048 + 3 tokens.  The line also carries the sweep over quantum 128..8192.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--quantum Q] [--workload NAME]
  python bench.py --impl reference ...     # the fp64 CPU oracle on the same workload

Under torchrun (N > 1) every rank runs its own independent layer step on its own GPU with its
own token batch (replicas, weak scaling; no collective on the data path); time is the max over
ranks and value is all ranks' tokens over that time.
"""
from __future__ import annotations

import argparse
import hashlib
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


def _times_the_oracle(argv) -> bool:
    """True for the reference arm and the CPU-baseline worker (both time the oracle on one core)."""
    if "--cpu-worker" in argv or "--impl=reference" in argv:
        return True
    return any(a == "--impl" and b == "reference" for a, b in zip(argv, argv[1:]))


# BLAS reads its thread count when it loads, so the one-core pin precedes the numpy import.
if _times_the_oracle(sys.argv[1:]):
    for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_var] = "1"

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE layer tokens/s vs prefill quantum (1 GB300); % of HBM/tensor roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal GB300 figures, reported beside the measured-peak fractions: HBM3e ~8 TB/s, dense bf16
# 2.25 PFLOP/s.  The measured copy rate and cuBLAS rate are the denominators of `frac`.
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0


def nominal_frac(alg_bytes: float, flops: float, seconds: float) -> float:
    """Fraction of the nominal roofline max(bytes / 8 TB/s, flops / 2.25 PF) reached in `seconds`."""
    t = max(alg_bytes / (NOMINAL_HBM_GBS * 1e9), flops / (NOMINAL_BF16_TFLOPS * 1e12))
    return round(t / seconds, 4)


# ----------------------------------------------------------------------------------------------
# distributed helpers (also exercised by the CPU gloo test)
# ----------------------------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own token batch (weights are the same layer on every rank)."""
    return base + 1000003 * rank


# ----------------------------------------------------------------------------------------------
# peaks, clocks, roofline bookkeeping
# ----------------------------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_path: str | None = None):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.log_path = log_path

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        if self.log_path:
            with open(self.log_path, "w") as fh:
                fh.write(self.FIELDS + "\n" + "\n".join(self.lines) + "\n")
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def layer_bytes_flops(w: synth.Workload, counts: np.ndarray) -> dict:
    """Algorithmic bytes and FLOPs of one layer step (touched experts only)."""
    s = w.spec
    touched = int((counts > 0).sum())
    wbytes = 2.0 if s.wdtype == "bf16" else 0.5 + 1.0 / 32.0
    expert = 3.0 * s.d * s.f * wbytes
    shared = 3.0 * s.d * s.f_s * 2.0 * s.n_shared
    router = s.d * s.E * 4.0 + s.E * 4.0
    act = w.T * s.d * 2.0 * 2 + w.T * s.k * 8.0
    flops = 2.0 * w.T * s.d * s.E + 6.0 * w.T * s.k * s.d * s.f + 6.0 * w.T * s.n_shared * s.d * s.f_s
    return {"touched": touched, "bytes": touched * expert + shared + router + act, "flops": flops,
            "gateup_bytes": touched * 2.0 * s.d * s.f * wbytes + 2.0 * s.d * s.f_s * 2.0 * s.n_shared
            + w.T * s.d * 2.0 + (w.T * s.k * s.f + w.T * s.n_shared * s.f_s) * 2.0,
            "down_bytes": touched * s.d * s.f * wbytes + s.d * s.f_s * 2.0 * s.n_shared
            + (w.T * s.k * s.f + w.T * s.n_shared * s.f_s) * 2.0 + (w.T * s.k + (w.T if s.n_shared else 0)) * s.d * 2.0,
            "weight_bytes": touched * expert + shared}


def kernel_alg_bytes(name: str, w: synth.Workload, counts: np.ndarray):
    """Algorithmic bytes of one launch of the named kernel (compulsory reads + writes)."""
    s = w.spec
    touched = int((counts > 0).sum())
    wb = 2.0 if s.wdtype == "bf16" else 0.5 + 1.0 / 32.0
    R = w.T * s.k
    h_r, h_s = R * s.f * 2.0, w.T * s.n_shared * s.f_s * 2.0
    y_r, y_s = R * s.d * 2.0, (w.T * s.d * 2.0 if s.n_shared else 0.0)
    sh_gu, sh_dn = 2.0 * s.d * s.f_s * 2.0 * s.n_shared, s.d * s.f_s * 2.0 * s.n_shared
    x = w.T * s.d * 2.0
    table = {
        "tc_gateup": touched * 2.0 * s.d * s.f * wb + sh_gu + x + h_r + h_s,
        "tc_down": touched * s.d * s.f * wb + sh_dn + h_r + h_s + y_r + y_s,
        "fp4_gateup": touched * 2.0 * s.d * s.f * wb + x + h_r,
        "fp4_down": touched * s.d * s.f * wb + h_r + y_r,
        "tc_gateup_shared": sh_gu + x + h_s,
        "tc_down_shared": sh_dn + h_s + y_s,
        "combine": y_r + y_s + x + R * 8.0,
        # the one-launch small step: the whole layer (router, touched and shared weights, x, out)
        "layer_small": touched * 3.0 * s.d * s.f * wb + sh_gu + sh_dn + s.d * s.E * 4.0 + 2.0 * x + R * 8.0,
    }
    return table.get(name)


# The sources a kernel's DRAM traffic depends on: its own file, the shared device helpers, the
# plan code that picks its launch shape and the weight layouts it reads.
_COMMON_SOURCES = ("common.cuh", "kernels.h", "api.cu", "repack.cu")
KERNEL_SOURCES = {
    "tc_gateup": ("gemm_tc.cu",), "tc_down": ("gemm_tc.cu",),
    "tc_gateup_shared": ("gemm_tc.cu",), "tc_down_shared": ("gemm_tc.cu",),
    "fp4_gateup": ("gemm_fp4.cu",), "fp4_down": ("gemm_fp4.cu",),
    "combine": ("combine.cu",),
    "layer_small": ("layer_small.cu", "topk.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources of one kernel (KERNEL_SOURCES plus the shared ones)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_batches_gb300", "csrc")
    for name in sorted(set(KERNEL_SOURCES[kernel] + _COMMON_SOURCES)):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_key(kernel: str, w: synth.Workload) -> str:
    return f"{kernel}@{w.name}_T{w.T}"


def committed_traffic(kernel: str, w: synth.Workload):
    """dram bytes per launch of `kernel` on workload `w` from the committed ncu summary, if it
    was taken on the kernel's current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            tr = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = tr.get(traffic_key(kernel, w))
    if not ent or kernel not in KERNEL_SOURCES or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------
def workload_from_args(args, seed=0) -> synth.Workload:
    return synth.workload(args.workload, quantum=args.quantum, seed=seed)


def upload_plan(w: synth.Workload, T_max: int):
    import torch
    from decode_batches_gb300 import MoePlan

    s = w.spec
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bf = lambda a: dev(a).view(torch.bfloat16)
    plan = MoePlan(s.E, s.k, s.d, s.f, s.n_shared, s.wdtype)
    ex = w.experts()
    b = w.router_bias()
    if s.wdtype == "bf16":
        plan.set_weights(dev(w.router_weight()), dev(b) if b is not None else None, bf(ex.gate), bf(ex.up), bf(ex.down))
    else:
        plan.set_weights(dev(w.router_weight()), dev(b) if b is not None else None, dev(ex.gate), dev(ex.up),
                         dev(ex.down), dev(ex.gate_scale), dev(ex.up_scale), dev(ex.down_scale))
    sh = w.shared()
    if sh is not None:
        plan.set_shared(s.f_s, bf(sh[0]), bf(sh[1]), bf(sh[2]))
    plan.allocate_workspace(T_max)
    w.drop_cache()          # host copies of the weights are no longer needed
    return plan


def time_forward(plan, x, n_prefill, steps, warmup, world, timing=False):
    """Device time of `steps` forwards (CUDA events on the launching stream), max over ranks."""
    import torch
    st = torch.cuda.current_stream()
    out = torch.empty_like(x)
    for _ in range(warmup):
        plan.forward(x, n_prefill, out=out)
    plan.timing_report()  # discard warm-up events
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    if timing:
        plan.enable_timing(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        plan.forward(x, n_prefill, out=out)
    e1.record(st)
    torch.cuda.synchronize()
    plan.enable_timing(False)
    ms = e0.elapsed_time(e1)
    kernels = plan.timing_report() if timing else {}
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    return reduce_max(ms, world, device="cuda" if world > 1 else None) / steps, kernels, out


def time_forward_cold(plan, x, n_prefill, steps, warmup, world):
    """Median device time of one forward with L2 flushed before each step: a buffer of twice the
    L2 size is written between steps, outside the step's CUDA-event pair, so the step's weights
    come from HBM.  Returns (median ms, max over ranks of the median)."""
    import torch
    st = torch.cuda.current_stream()
    l2 = int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 0)) or (126 << 20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.int32, device="cuda")
    out = torch.empty_like(x)
    for _ in range(warmup):
        plan.forward(x, n_prefill, out=out)
    times = []
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(i)
        evs[i][0].record(st)
        plan.forward(x, n_prefill, out=out)
        evs[i][1].record(st)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    med = statistics.median(times)
    del flush
    return reduce_max(med, world, device="cuda" if world > 1 else None)


def time_e2e(plan, x_host, n_prefill, steps, warmup, world):
    """Same metric through host buffers: every step copies its input from pinned host memory to
    the device, runs the layer and copies its output back to pinned host memory.  The two copies
    run on their own streams with double-buffered device tensors, so step i+1's input copy and
    step i-1's output copy overlap step i's layer, as a serving loop would; every copy of every
    timed step is inside the timed region."""
    import torch
    st = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    x_dev = [torch.empty(x_host.shape, dtype=x_host.dtype, device="cuda") for _ in range(2)]
    out_dev = [torch.empty_like(x_dev[0]) for _ in range(2)]
    out_host = [torch.empty(x_host.shape, dtype=x_host.dtype, pin_memory=True) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n, first):
        for i in range(n):
            b = i % 2
            reuse = not (first and i < 2)
            with torch.cuda.stream(h2d):
                if reuse:
                    h2d.wait_event(ev_done[b])     # step i-2's layer has read x_dev[b]
                x_dev[b].copy_(x_host, non_blocking=True)
                ev_in[b].record(h2d)
            st.wait_event(ev_in[b])
            if reuse:
                st.wait_event(ev_out[b])           # step i-2's output has left out_dev[b]
            plan.forward(x_dev[b], n_prefill, out=out_dev[b])
            ev_done[b].record(st)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_done[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                ev_out[b].record(d2h)

    run(warmup, True)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    h2d.wait_event(e0)
    d2h.wait_event(e0)
    run(steps, True)
    st.wait_stream(h2d)
    st.wait_stream(d2h)  # the last output copy is inside the timed region
    e1.record(st)
    torch.cuda.synchronize()
    ms = reduce_max(e0.elapsed_time(e1), world, device="cuda" if world > 1 else None) / steps
    nbytes = x_host.numel() * x_host.element_size()
    return ms, nbytes, nbytes


def routing_counts(plan, x):
    _, ids, _ = plan.route(x, want_logits=False)
    counts, _, _, _ = plan.permute(ids)
    return counts.cpu().numpy()


def run_gpu(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks["bf16_tflops"])

    w = workload_from_args(args, seed=rank_seed(0, rank) if world > 1 else 0)
    x_np = w.x()
    T = w.T
    sweep_q = [q for q in synth.QUANTA] if (args.workload == "mixed" and not args.no_sweep) else []
    serve = args.workload == "mixed" and not args.no_extra
    T_max = max([T] + [q + 3 for q in sweep_q] + ([SERVE_CAP_MAX + SERVE_DECODE_ROWS] if serve else []))
    # weights: identical layer on every rank (seed 0); tokens per rank from the rank's seed
    wl_weights = synth.workload(args.workload, quantum=args.quantum, seed=0)
    plan = upload_plan(wl_weights, T_max)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    x = dev(x_np).view(torch.bfloat16)
    counts = routing_counts(plan, x)
    bf = layer_bytes_flops(w, counts)

    clocks = ClockSampler(local, args.clocks_log)
    clocks.start()
    # timed region: K steps, nothing recorded between the layer's kernels
    ms, _, _ = time_forward(plan, x, w.n_prefill, args.steps, args.warmup, world)
    clk = clocks.stop()
    # the same step with L2 flushed before each step (median), outside the headline's timed region
    cold_ms = time_forward_cold(plan, x, w.n_prefill, max(20, min(args.steps, 200)), 3, world)
    # per-kernel durations: a second timed region with CUDA events around every launch (the
    # events serialise the launches, so this region is not the one `value` comes from)
    _, kernels, _ = time_forward(plan, x, w.n_prefill, max(20, args.steps // 4), 3, world, timing=True)
    launches_per_step = plan.last_launch_count()

    tokens_per_s = world * T / (ms * 1e-3)
    t_roof = max(bf["bytes"] / (hbm * 1e9), bf["flops"] / (tflops * 1e12))
    # dominant kernel by total time inside the timed region
    dom = max(kernels.items(), key=lambda kv: kv[1][1]) if kernels else None
    roofline = None
    if dom:
        name, (n, tot_ms) = dom
        per_launch_s = tot_ms / n * 1e-3
        alg, bound = kernel_alg_bytes(name, w, counts), "hbm"
        if alg is None:
            alg = bf["bytes"]
        achieved = alg / per_launch_s / 1e9
        tr = committed_traffic(name, w)
        roofline = {"bound": bound, "kernel": name, "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(achieved / hbm, 4), "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                    "traffic": tr["bytes_per_launch"] if tr else None,
                    "algorithmic_bytes": alg, "launch_us": round(per_launch_s * 1e6, 2),
                    "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else peak_src}

    # e2e through host buffers
    x_host = torch.from_numpy(np.ascontiguousarray(x_np)).view(torch.bfloat16).pin_memory()
    e2e_ms, h2d, d2h = time_e2e(plan, x_host, w.n_prefill, max(3, args.steps // 4), max(3, args.warmup), world)

    sweep = []
    for q in sweep_q:
        wq = synth.workload("mixed", quantum=q, seed=rank_seed(0, rank) if world > 1 else 0)
        xq = dev(wq.x()).view(torch.bfloat16)
        cq = routing_counts(plan, xq)
        bq = layer_bytes_flops(wq, cq)
        msq, _, _ = time_forward(plan, xq, wq.n_prefill, max(20, min(args.steps, 400)), max(3, args.warmup), world)
        _, kq, _ = time_forward(plan, xq, wq.n_prefill, max(20, min(args.steps, 100)), 3, world, timing=True)
        tq = max(bq["bytes"] / (hbm * 1e9), bq["flops"] / (tflops * 1e12))
        sweep.append({"quantum": q, "T": wq.T, "tokens_per_s": round(world * wq.T / (msq * 1e-3), 1),
                      "ms_per_step": round(msq, 5), "touched_experts": bq["touched"],
                      "roofline_frac": round(tq / (msq * 1e-3), 4),
                      "roofline_frac_nominal": nominal_frac(bq["bytes"], bq["flops"], msq * 1e-3),
                      "bound": "hbm" if bq["bytes"] / (hbm * 1e9) >= bq["flops"] / (tflops * 1e12) else "tensor",
                      "kernel_us": {k: round(v[1] / v[0] * 1e3, 2) for k, v in kq.items()}})

    serving = serving_runs(plan, world, rank) if serve else None

    extra = {}
    if not args.no_extra and args.workload == "mixed":
        # the other configurations of the layer: 4-token decode on the same plan; the 4-bit Zipf
        # step and the 6-row verify batch on a 384-expert 4-bit plan
        extra["decode_T4"] = measure_workload(plan, synth.workload("decode", seed=rank_seed(0, rank) if world > 1 else 0),
                                              hbm, tflops, world, args)
        del plan
        torch.cuda.empty_cache()
        fp4_plan = upload_plan(synth.workload("fp4_zipf", seed=0), 2051)
        extra["fp4_zipf_T2051"] = measure_workload(fp4_plan, synth.workload("fp4_zipf", seed=rank_seed(0, rank) if world > 1 else 0),
                                                   hbm, tflops, world, args)
        extra["verify_8x6_T48"] = measure_workload(fp4_plan, synth.workload("verify", seed=rank_seed(0, rank) if world > 1 else 0),
                                                   hbm, tflops, world, args, committed=(48, 8))
        del fp4_plan
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_subprocess(args)

    line = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.spec.wdtype == "bf16" else "bf16 activations, mxfp4 weights",
        "data": "synthetic (seeded counter-based normals; random-init weights of the layer's shape)",
        "config": bench_config(w, args, world),
        "layer_roofline": {"bytes": bf["bytes"], "flops": bf["flops"], "t_roofline_us": round(t_roof * 1e6, 2),
                           "frac": round(t_roof / (ms * 1e-3), 4), "hbm_gbs": hbm, "bf16_tflops": tflops,
                           "peak_source": peak_src, "frac_nominal": nominal_frac(bf["bytes"], bf["flops"], ms * 1e-3),
                           "touched_experts": bf["touched"], "weight_bytes": bf["weight_bytes"],
                           "weight_bytes_per_token": round(bf["weight_bytes"] / T, 1),
                           "cold_l2": {"ms_per_step_median": round(cold_ms, 5),
                                       "frac": round(t_roof / (cold_ms * 1e-3), 4),
                                       "frac_nominal": nominal_frac(bf["bytes"], bf["flops"], cold_ms * 1e-3)}},
        "roofline": roofline,
        "kernels": {k: {"launches": v[0], "total_ms": round(v[1], 4), "avg_us": round(v[1] / v[0] * 1e3, 2)}
                    for k, v in kernels.items()},
        "e2e": {"value": round(world * T / (e2e_ms * 1e-3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": launches_per_step * args.steps,
        "launches_per_step": launches_per_step,
        "clocks": clk,
        "sweep": sweep,
        "workloads": extra,
        "serving": serving,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


SERVE_DECODE_ROWS = 3      # generating sessions riding along in every prefill call (c2's mix)
SERVE_CAP_MAX = 4096       # the engine's default prefill_cap


def serving_runs(plan, world: int, rank: int, reps: int = 3) -> dict:
    """Whole prompts prefilled through the step composer (the library's moe_compose_prefill), one
    layer call per composed call with SERVE_DECODE_ROWS decode rows appended while sessions are
    generating -- the one-layer analogue of the "moe-prefill-quantum" page's Figure 1 / Table 3
    (a 20,000-token cold prefill per quantum, three sessions decoding), Table 11 (an 8,478-token
    span at a context of 81,920 cut at boundaries 4096 / 3072 / 2560) and Table 1's first row
    (nothing generating: the quantum is not used).  Time per prompt: CUDA events around all its
    calls, median of `reps` after one warm-up run."""
    import torch
    from decode_batches_gb300 import compose_prefill
    src = synth.workload("mixed", quantum=SERVE_CAP_MAX, seed=rank_seed(7, rank))
    x_all = torch.from_numpy(np.ascontiguousarray(src.x())).cuda().view(torch.bfloat16)
    out = torch.empty_like(x_all)
    st = torch.cuda.current_stream()

    def run(start, n, q, active, cap):
        calls = compose_prefill(start, n, q, active, cap)
        dec = SERVE_DECODE_ROWS if active else 0
        times = []
        for r in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _, c, _ in calls:
                plan.forward(x_all[:c + dec], n_prefill=c, out=out[:c + dec])
            e1.record(st)
            torch.cuda.synchronize()
            if r:
                times.append(e0.elapsed_time(e1))
        ms = reduce_max(statistics.median(times), world, device="cuda" if world > 1 else None)
        return {"prompt_tokens": n, "start_pos": start, "quantum": q, "generation_active": active,
                "prefill_cap": cap, "calls": len(calls), "mean_call": round(n / len(calls), 1),
                "decode_rows_per_call": dec, "ms": round(ms, 3),
                "prefill_tokens_per_s": round(world * n / (ms * 1e-3), 1)}

    fig1 = [run(0, 20000, q, True, SERVE_CAP_MAX) for q in synth.QUANTA]
    t11 = [run(81920, 8478, 2048, True, cap) for cap in (4096, 3072, 2560)]
    idle = [run(0, 20000, q, False, SERVE_CAP_MAX) for q in (128, 2048)]
    return {"prefill_vs_quantum": fig1, "calls_vs_boundary": t11, "no_generation": idle}


def measure_workload(plan, w: synth.Workload, hbm: float, tflops: float, world: int, args, committed=None) -> dict:
    """tokens/s, roofline and per-kernel times of one more workload on an uploaded plan."""
    import torch
    x = torch.from_numpy(np.ascontiguousarray(w.x())).cuda().view(torch.bfloat16)
    counts = routing_counts(plan, x)
    b = layer_bytes_flops(w, counts)
    steps = max(50, min(args.steps, 1000))
    ms_warm, _, _ = time_forward(plan, x, w.n_prefill, steps, max(3, args.warmup), world)
    ms = time_forward_cold(plan, x, w.n_prefill, max(50, min(args.steps, 200)), max(3, args.warmup), world)
    _, k, _ = time_forward(plan, x, w.n_prefill, max(20, steps // 4), 3, world, timing=True)
    t_hbm, t_tc = b["bytes"] / (hbm * 1e9), b["flops"] / (tflops * 1e12)
    out = {"workload": workload_desc(w), "T": w.T, "tokens_per_s": round(world * w.T / (ms * 1e-3), 1),
           "ms_per_step": round(ms, 5), "timing": "median of per-step CUDA-event times, L2 flushed before each step",
           "ms_per_step_back_to_back": round(ms_warm, 5), "touched_experts": b["touched"], "alg_bytes": b["bytes"],
           "flops": b["flops"], "bound": "hbm" if t_hbm >= t_tc else "tensor",
           "roofline_frac": round(max(t_hbm, t_tc) / (ms * 1e-3), 4),
           "roofline_frac_nominal": nominal_frac(b["bytes"], b["flops"], ms * 1e-3),
           "hbm_frac": round(b["bytes"] / (ms * 1e-3) / (hbm * 1e9), 4),
           "hbm_frac_nominal": round(b["bytes"] / (ms * 1e-3) / (NOMINAL_HBM_GBS * 1e9), 4),
           "launches_per_step": plan.last_launch_count(),
           "kernel_us": {n: round(v[1] / v[0] * 1e3, 2) for n, v in k.items()}}
    if committed:
        # weight bytes streamed per committed token: every verify row accepted / one per sequence
        out["weight_bytes_per_committed_token"] = {f"{c}_committed": round(b["weight_bytes"] / c, 1) for c in committed}
    return out


def bench_config(w: synth.Workload, args, world: int) -> dict:
    """The `config` object of the JSON line; identical for this arm and the reference arm."""
    s = w.spec
    return {"workload": workload_desc(w), "T": w.T, "n_prefill": w.n_prefill,
            "quantum": args.quantum if args.workload == "mixed" else None, "d_model": s.d, "experts": s.E,
            "top_k": s.k, "d_ff": s.f, "n_shared": s.n_shared, "d_ff_shared": s.f_s, "weights": s.wdtype,
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "l2": "inputs larger than L2: the touched expert weights (about 1.6 GB at the mixed step's quanta, "
                  "2.6 GB at the 4-bit layer) stream from HBM every step; the small-T rows of `workloads` "
                  "also flush L2 (a buffer of twice its size) before each timed step"}


def workload_desc(w: synth.Workload) -> str:
    s = w.spec
    if w.name.startswith("mixed"):
        return (f"mixed prefill+decode step: quantum {w.n_prefill} + {w.T - w.n_prefill} decode tokens (T={w.T}), "
                f"d_model {s.d}, {s.E} experts top-{s.k}, d_ff {s.f}, {s.n_shared} shared d_ff {s.f_s}, {s.wdtype}")
    return f"{w.name}: T={w.T}, d_model {s.d}, {s.E} experts top-{s.k}, d_ff {s.f}, shared {s.n_shared}x{s.f_s}, {s.wdtype}"


# ----------------------------------------------------------------------------------------------
# CPU oracle arm (baseline and --impl reference)
# ----------------------------------------------------------------------------------------------
def oracle_tokens(w: synth.Workload, rows: np.ndarray) -> float:
    """Run the fp64 oracle layer on the given token rows; returns seconds."""
    import oracle
    ex = w.experts()
    dec = oracle.DecodedExperts(ex.gate, ex.up, ex.down, ex.gate_scale, ex.up_scale, ex.down_scale)
    t0 = time.perf_counter()
    oracle.moe_layer(w.x()[rows], w.router_weight(), w.router_bias(), w.spec.k, dec, w.shared())
    return time.perf_counter() - t0


CPU_BASELINE_SECONDS = 15.0   # oracle work the default CPU baseline aims at


def cpu_worker(args):
    """Child process (BLAS pinned to one thread): time the oracle on a bounded token sample.
    --sample N fixes the number of tokens; 0 sizes it to about CPU_BASELINE_SECONDS of oracle
    work, capped at the whole step: calibration runs grow 4x from 64 tokens until one takes a
    quarter of that (the oracle's per-expert cost amortises over the tokens, so a small
    calibration overestimates the cost per token)."""
    w = workload_from_args(args)
    rng = np.random.default_rng(123)
    order = rng.permutation(w.T)
    oracle_tokens(w, order[:1])            # warm (page in weights, import)
    if args.sample > 0:
        n = min(args.sample, w.T)
    else:
        n = min(64, w.T)
        while True:
            dt = oracle_tokens(w, np.sort(order[:n]))
            if n >= w.T or dt >= CPU_BASELINE_SECONDS / 4:
                break
            n = min(w.T, 4 * n)
        n = int(min(w.T, max(n, n * CPU_BASELINE_SECONDS / max(dt, 1e-6))))
    rows = np.sort(order[:n])
    dt = oracle_tokens(w, rows)
    print(json.dumps({"value": n / dt, "seconds": dt, "tokens": n, "T": w.T}))


def cpu_baseline_subprocess(args) -> dict | None:
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               RANK="0", WORLD_SIZE="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--workload", args.workload, "--quantum",
           str(args.quantum), "--sample", str(args.cpu_sample)]
    try:
        res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        out = json.loads(res.stdout.strip().splitlines()[-1])
    except Exception as exc:  # noqa: BLE001 - reported, never fatal for the GPU line
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "error": str(exc)[:200]}
    return {"value": round(out["value"], 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{out['tokens']} of the step's {out['T']} tokens (seeded), full fp64 layer per token "
                      f"(router, top-k, grouping, expert FFNs, combine, shared expert); "
                      f"{out['seconds']:.1f} s single-threaded numpy"}


def run_reference(args):
    """--impl reference: the fp64 oracle timed as it stands on the host cores, rank 0 only."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workload_from_args(args)
    rng = np.random.default_rng(7)
    # Calibrate the oracle's cost per token on samples growing 4x from 64 tokens until one takes
    # about a second (its per-expert work amortises over the tokens of a step, so one token alone
    # overstates the cost), then size each step's sample so the whole run takes about 2 minutes:
    # at the driver's few steps that is the whole step, as in the CPU baseline.
    order = rng.permutation(w.T)
    oracle_tokens(w, order[:1])
    n = min(64, w.T)
    while True:
        dt = oracle_tokens(w, np.sort(order[:n]))
        if n >= w.T or dt >= 1.0:
            break
        n = min(w.T, 4 * n)
    per_token = dt / n
    budget = 120.0 / max(1, args.steps + args.warmup)
    per_step = int(max(1, min(w.T, budget / max(per_token, 1e-6))))
    times, toks = [], 0
    for i in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(w.T, size=per_step, replace=False))
        dt = oracle_tokens(w, rows)
        if i >= args.warmup:
            times.append(dt)
            toks += per_step
    total = sum(times)
    value = toks / total
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / len(times) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based normals; random-init weights of the layer's shape)",
        "config": bench_config(w, args, world),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "kind": "oracle", "cores": 1,
                         "sample": f"{per_step} seeded tokens of the {w.T}-token step per timed step"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixed", choices=["tiny", "decode", "mixed", "fp4_zipf", "verify"])
    ap.add_argument("--quantum", type=int, default=2048)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the decode, 4-bit and verify workloads")
    ap.add_argument("--cpu-sample", type=int, default=0,
                    help="tokens of the CPU-baseline sample (0: about 15 s of oracle work, at most the whole step)")
    ap.add_argument("--clocks-log", default=None, help="write the nvidia-smi samples of the timed region here")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--sample", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.cpu_worker:
        return cpu_worker(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    main()
