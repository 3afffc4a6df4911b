#!/usr/bin/env python
"""Benchmark of the PRISM memory-recurrence forward on GB300.

Metric: tokens/s of one PRISM layer forward (B*T tokens, all heads) at the
16K-token sequential-recommendation shape (B=2, H=4, T=16384, dk=dv=64, L=4,
bf16 io), plus the achieved fraction of the roofline of the binding resource.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one prism_forward over the whole synthetic batch (inputs resident in
HBM).  L2 is flushed (a 512 MiB write, then a 512 MiB read, so that no dirty line of
the flush is written back inside the timed region) before every timed step and the step is
timed alone with CUDA events on the launch stream.  N > 1 runs one independent
replica per GPU (the path has no exchange step), launched by torchrun; rank 0
prints one JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "PRISM layer fwd tokens/s on 1 GB300 (T=16K) + % of HBM/tensor roofline"
NONLINEAR_METRIC = "PRISM layer fwd tokens/s, non-linear residual variant + % of HBM roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
THROTTLE_BITS = {  # nvidia-smi clocks_event_reasons bit masks
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
    0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
    0x80: "hw_power_brake_slowdown", 0x100: "display_clocks_setting",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="default seqrec_16k (forward) or decode_lm130m (decode)")
    ap.add_argument("--mode", choices=["forward", "decode", "nonlinear", "project", "backward"], default="forward",
                    help="forward: prism_forward over whole sequences (the headline); decode: one "
                         "prism_decode_step (one token per sequence) over a serving batch; nonlinear: "
                         "prism_forward_nonlinear (the non-linear residual variant) over whole sequences; "
                         "project: prism_project (the block's input projections); backward: prism_backward "
                         "(the cotangents of every input) over whole sequences")
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 portable fp32 kernels, 2 tensor-core path")
    ap.add_argument("--nonlinear", action="store_true",
                    help="backward mode: prism_backward_nonlinear (the non-linear residual chain's cotangents)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override the workload's T (a smaller case of the same shape, e.g. for a profiler)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target length of the CPU-baseline sample")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------------------
# algorithmic work of the path, per (token, head)
def alg_bytes_per_token_head(w, nonlinear=False):
    io = 2 if w.dtype == "bf16" else 4
    if nonlinear:  # gains p (R dv, io dtype) in place of eta
        return io * (2 * w.dk + 2 * w.dv + w.R * w.dk + w.R * w.dv) + 4 * (2 + w.R)
    return io * (2 * w.dk + 2 * w.dv + w.R * w.dk) + 4 * (2 + 2 * w.R)


def alg_flops_per_token_head(w):
    # sequential form: S k, rank-1 correction, L outer products, S q  ->  2 d^2 (L + 3) for dk = dv = d
    return 2 * w.dk * w.dv * (w.L + 3)


def kernel_alg_bytes(name, w, nonlinear=False):
    """Bytes a kernel must move at minimum (each of its inputs read once, each output written
    once), for one launch over the whole workload."""
    io = 2 if w.dtype == "bf16" else 4
    th = w.B * w.H * w.T
    nc = -(-w.T // 64)
    chunks = w.B * w.H * nc
    R = w.R
    q = k = th * w.dk * io
    v = out = th * w.dv * io
    u = th * R * w.dk * io
    gates = th * 4 * (2 + 2 * R)
    X = th * R * w.dv * 4
    lam = th * 4
    Tm = chunks * 64 * 64 * 4
    W = th * w.dk * 4
    Up = Vt = th * w.dv * 4
    S0 = chunks * w.dv * w.dk * 4
    p_or_eta = th * R * w.dv * io if nonlinear else th * 4 * R
    table = {
        "map_chunks": q + k + v + u + gates,      # every input read once (the maps are its own output)
        "map_scan": out,                          # the outputs written once (the maps are read back)
        "map_compose": chunks * 2 * w.dk * w.dv * 2,  # long sequences: every chunk's A_c and B_c read once
        "map_carry": w.B * w.H * w.dk * w.dv * 4,     # the segments' start states (a floor: one state)
        "simt_prep": v + th * 4 * R + p_or_eta + X,
        "simt_chunk_solve": k + th * 8 + lam + Tm,
        "simt_wy": k + v + th * 4 + u + X + lam + Tm + W + Up,
        "simt_state": k + u + X + lam + W + Up + S0 + Vt,
        "simt_out": q + k + u + X + lam + S0 + Vt + out,
    }
    if nonlinear:
        gates = th * 4 * (2 + R) + th * R * w.dv * io
    return table.get(name, q + k + v + u + gates + out)


# the source files each kernel is built from (its own translation unit and the headers it uses)
ROOFLINE_TARGET = 0.5  # fraction of the binding resource's measured roofline the forward aims for

KERNEL_SOURCES = {
    "project": ("prism_project.cu", "prism_project.h", "tc_ptx.h", "prism_internal.h"),
    "tc_": ("prism_tc.cu", "tc_ptx.h", "prism_internal.h"),
    "map_": ("prism_map.cu", "tc_util.h", "tc_ptx.h", "prism_internal.h"),
    "decode": ("prism_state.cu", "tc_ptx.h", "prism_internal.h"),
    "simt_": ("prism_simt.cu", "prism_internal.h"),
    "bwd_maps": ("prism_bwd_tc.cu", "tc_util.h", "tc_ptx.h", "prism_internal.h"),
    "bwd_chunk": ("prism_bwd_tc.cu", "tc_util.h", "tc_ptx.h", "prism_internal.h"),
    "bwd_grad": ("prism_bwd_tc.cu", "tc_util.h", "tc_ptx.h", "prism_internal.h"),
    "bwd_": ("prism_backward.cu", "tc_util.h", "tc_ptx.h", "prism_internal.h"),
}


def traffic_from_profiles(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    source of that kernel (the summary records the digest of the kernel's source files);
    else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != source_digest(kernel):
        return None
    return float(m.group(1))


def source_digest(kernel):
    files = next((f for prefix, f in KERNEL_SOURCES.items() if kernel.startswith(prefix)), None)
    csrc = os.path.join(ROOT, "ssm_sequence_layer_gb300", "csrc")
    if files is None:
        files = sorted(fn for fn in os.listdir(csrc) if fn.endswith((".cu", ".h")))
    h = hashlib.sha256()
    for fn in files:
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------------------------------------
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", "200"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 3:
                try:
                    self.samples.append((float(parts[0]), float(parts[1]), int(parts[2], 16)))
                except ValueError:
                    pass

    def stop(self):
        time.sleep(0.25)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [s[0] for s in self.samples]
        reasons = set()
        for s in self.samples:
            for bit, name in THROTTLE_BITS.items():
                if s[2] & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(s[1] for s in self.samples),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
class L2Flush:
    """Evicts L2 (129 MB on GB300) between timed steps: a 512 MiB write, then a 512 MiB read of
    another buffer, so that the lines the write leaves dirty are written back before the timed
    region starts rather than inside it."""

    DESCRIPTION = "flushed before every timed step: 512 MiB written, then 512 MiB of another buffer read"

    def __init__(self):
        import torch
        n = 512 * 1024 * 1024 // 4
        self.w = torch.empty(n, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.sink = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    from ssm_sequence_layer_gb300.replicas import barrier as _barrier
    _barrier(world)


def max_over_ranks(x, world):
    from ssm_sequence_layer_gb300.replicas import max_over_ranks as _max
    return _max(x, world, device="cuda")


def oracle_sample(w, inp, seconds_target, nthreads, p_gain=None):
    """Time the oracle on the first Ts tokens of every sequence, Ts sized so the run takes
    about `seconds_target` seconds.  Returns (tokens/s, Ts, seconds, oracle output [B,H,Ts,dv])."""
    from oracle import prism_oracle

    def run(Ts):
        sub = {k: (v[:, :, :Ts] if hasattr(v, "shape") and k != "conv_w" else v) for k, v in inp.items()}
        t0 = time.perf_counter()
        res = prism_oracle.forward(sub["q"], sub["k"], sub["v"], sub["beta"], sub["alpha"], sub["u"], sub["gamma"],
                                   sub["eta"], sub["conv_w"], sub["L"], nthreads=nthreads,
                                   p_gain=None if p_gain is None else p_gain[:, :, :Ts])
        return time.perf_counter() - t0, res["out"]

    Ts = min(w.T, 256)
    dt, _ = run(Ts)
    Ts = int(min(w.T, max(Ts, Ts * seconds_target / max(dt, 1e-3))))
    dt, ref = run(Ts)
    return w.B * Ts / dt, Ts, dt, ref


def parity_error(out, ref, bf16_out):
    """max |o - o_ref| / rms(o_ref) over the compared outputs; for a bf16 output each element is
    first allowed the half-ulp its own rounding to bf16 costs (at the larger of |o| and |o_ref|)."""
    import numpy as np
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    diff = np.abs(out - ref)
    if bf16_out:
        a = np.maximum(np.abs(out), np.abs(ref))
        half_ulp = np.where(a > 0, np.exp2(np.floor(np.log2(np.maximum(a, 1e-300))) - 8), 0.0)
        diff = np.maximum(diff - half_ulp, 0.0)
    return float(np.max(diff) / max(rms, 1e-300))


def cpu_threads(w):
    return max(1, min(len(os.sched_getaffinity(0)), w.B * w.H))


def cpu_model():
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu, which also names Arm cores)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def host_info(nthreads):
    """Threads the oracle used, the cores this process may run on, and the CPU model."""
    return {"cores": nthreads, "host_cores": len(os.sched_getaffinity(0)), "cpu_model": cpu_model()}


# ------------------------------------------------------------------------------------------------
def run_reference(args, w):
    """The oracle as the reference arm: each step is the oracle over the first Ts tokens of
    every sequence of the workload, on the host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from oracle import prism_oracle
    from ssm_sequence_layer_gb300.inputs import make_workload_inputs
    inp = make_workload_inputs(w)
    nthreads = cpu_threads(w)
    Ts = min(w.T, 1024)
    sub = {k: (v[:, :, :Ts].contiguous() if hasattr(v, "shape") and k != "conv_w" else v) for k, v in inp.items()}
    import numpy as np
    sub = {k: (v.double().numpy() if hasattr(v, "double") else v) for k, v in sub.items()}

    def step():
        prism_oracle.forward(sub["q"], sub["k"], sub["v"], sub["beta"], sub["alpha"], sub["u"], sub["gamma"],
                             sub["eta"], sub["conv_w"], sub["L"], nthreads=nthreads)

    for _ in range(max(args.warmup, 0)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = w.B * Ts * args.steps / dt
    sample = f"oracle over the first {Ts} tokens of all {w.B * w.H} (batch, head) sequences per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **{k: getattr(w, k) for k in ("B", "H", "T", "dk", "dv", "L")},
                   "io": w.dtype},
        "cpu_baseline": {"value": value, "unit": UNIT, **host_info(nthreads), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    del np
    return 0


def run_ours(args, w):
    import torch

    from ssm_sequence_layer_gb300 import binding as Bd
    from ssm_sequence_layer_gb300 import build as cuda_build
    from ssm_sequence_layer_gb300.inputs import make_gain, make_workload_inputs

    world, rank, local = dist_setup(args)
    if rank == 0:
        cuda_build.build()
    barrier(world)
    steps, warm = args.steps, max(args.warmup, 3)
    inp_cpu = make_workload_inputs(w, seed=0)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp_cpu.items()}
    out = torch.empty_like(dev["v"])
    stream = torch.cuda.current_stream()
    plan = Bd.Plan.for_inputs(dev, path=args.path if args.path else None)
    flush = L2Flush()
    nonlinear = args.mode == "nonlinear"
    p_cpu = make_gain(w.B, w.H, w.T, w.L, w.dv, dtype=w.dtype, seed=0) if nonlinear else None
    p_dev = p_cpu.cuda() if nonlinear else None

    def forward(inputs, p):
        if nonlinear:
            plan.forward_nonlinear(inputs, p, out=out, stream=stream)
        else:
            plan.forward(inputs, out, stream)

    for _ in range(warm):
        flush()
        forward(dev, p_dev)
    torch.cuda.synchronize()
    plan.last_device_status()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):  # the timed steps: no per-kernel events inside the forward
        flush()
        ev[i][0].record(stream)
        forward(dev, p_dev)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    plan.last_device_status()
    timed_out = out.detach().cpu()  # the output of the last timed step, checked against the oracle below
    step_ms = [a.elapsed_time(b) for a, b in ev]
    # per-kernel durations: the same number of forwards again, with CUDA events around every
    # kernel launch on the plan's stream (these runs are not part of the step time)
    plan.set_option(Bd.PRISM_OPT_TIMING, 1)
    per_kernel = {}
    launches = 0
    for i in range(steps):
        flush()
        forward(dev, p_dev)
        torch.cuda.synchronize()
        kt = plan.kernel_times()
        launches += len(kt)
        for name, ms in kt:
            per_kernel.setdefault(name, []).append(ms)
    plan.set_option(Bd.PRISM_OPT_TIMING, 0)
    plan.last_device_status()

    # the same forward replayed from a CUDA graph (L2 flushed before each replay, outside the
    # graph), and back-to-back forwards with a warm L2 -- reported beside the main figure
    graph_ms = None
    if not nonlinear:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.forward(dev, out, torch.cuda.current_stream())
        torch.cuda.synchronize()
        gms = []
        for i in range(steps + 3):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                gms.append(a.elapsed_time(b))
        plan.last_device_status()
        graph_ms = {"mean": sum(gms) / len(gms), "median": statistics.median(gms)}
        del g
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    forward(dev, p_dev)
    a.record(stream)
    for _ in range(steps):
        forward(dev, p_dev)
    b.record(stream)
    torch.cuda.synchronize()
    warm_ms = a.elapsed_time(b) / steps
    ms_local = sum(step_ms) / steps
    ms = max_over_ranks(ms_local, world)
    tokens_per_step = w.B * w.T
    value = tokens_per_step * world / (ms / 1e3)

    peaks, peak_kind = load_peaks()
    # dominant kernel: largest share of the measured kernel time
    tot = {n: sum(v) for n, v in per_kernel.items()}
    dom = max(tot, key=tot.get)
    dom_ms = tot[dom] / len(per_kernel[dom])
    dom_bytes = kernel_alg_bytes(dom, w, nonlinear)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    hbm = float(peaks["hbm_gbs"])
    path_bytes = alg_bytes_per_token_head(w, nonlinear) * w.B * w.H * w.T
    path_achieved = path_bytes / (ms_local / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                # the non-linear variant's counters are not the linear chain's (its gains add reads)
                "frac": achieved / hbm,
                "traffic": traffic_from_profiles(dom, w.name + ("_nonlinear" if nonlinear else "")),
                "alg_bytes_per_launch": dom_bytes, "kernel_ms": dom_ms, "peak_source": f"{peak_kind} hbm_gbs"}
    kernels = {n: {"ms_mean": tot[n] / len(per_kernel[n]), "share": tot[n] / sum(tot.values())} for n in tot}
    path_roofline = {"achieved": path_achieved, "unit": "GB/s", "frac": path_achieved / hbm,
                     "alg_bytes_per_step": path_bytes,
                     "tensor_frac": alg_flops_per_token_head(w) * w.B * w.H * w.T / (ms_local / 1e3) / 1e12
                     / float(peaks["bf16_tflops"])}

    # end to end through the host entry point (pinned host buffers, copies inside the timed region)
    e2e = None
    if not args.no_e2e and nonlinear:  # no host entry point: the inputs copied in, the output back
        host = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in inp_cpu.items() if k != "eta"}
        host_p = p_cpu.pin_memory()
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = host_p.numel() * host_p.element_size() + sum(v.numel() * v.element_size() for v in host.values()
                                                            if torch.is_tensor(v))
        d2h = hout.numel() * hout.element_size()
        dbuf = {k: (torch.empty_like(v, device="cuda") if torch.is_tensor(v) else v) for k, v in host.items()}
        dbuf["eta"] = None
        dp = torch.empty_like(host_p, device="cuda")
        e2e_ms = []
        for i in range(max(3, min(steps, 20)) + 2):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k, v in host.items():
                if torch.is_tensor(v):
                    dbuf[k].copy_(v, non_blocking=True)
            dp.copy_(host_p, non_blocking=True)
            forward(dbuf, dp)
            hout.copy_(out, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                e2e_ms.append(a.elapsed_time(b))
        e2e_ms_mean = max_over_ranks(sum(e2e_ms) / len(e2e_ms), world)
        e2e = {"value": tokens_per_step * world / (e2e_ms_mean / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_mean}
    elif not args.no_e2e:
        host = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in inp_cpu.items()}
        hout = torch.empty_like(host["v"]).pin_memory()
        h2d = sum(v.numel() * v.element_size() for k, v in host.items()
                  if torch.is_tensor(v) and (w.L > 1 or k not in ("u", "gamma", "eta")))
        d2h = hout.numel() * hout.element_size()
        for _ in range(2):
            plan.forward_host(host, hout, stream)
        e2e_ms = []
        for _ in range(max(3, min(steps, 20))):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            plan.forward_host(host, hout, stream)
            b.record(stream)
            torch.cuda.synchronize()
            e2e_ms.append(a.elapsed_time(b))
        e2e_ms_mean = max_over_ranks(sum(e2e_ms) / len(e2e_ms), world)
        e2e = {"value": tokens_per_step * world / (e2e_ms_mean / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_mean}

    cpu = None
    parity = parity_detail = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = cpu_threads(w)
        v, Ts, dt, ref = oracle_sample(w, inp_cpu, args.cpu_seconds, nthreads,
                                       p_gain=p_cpu.double().numpy() if nonlinear else None)
        cpu = {"value": v, "unit": UNIT, **host_info(nthreads), "kind": "oracle",
               "sample": f"fp64 oracle over the first {Ts} tokens of all {w.B * w.H} sequences ({dt:.1f} s)"}
        # the timed output against the oracle rows the baseline just computed (same inputs)
        got = timed_out[:, :, :Ts].double().numpy()
        bf16_out = timed_out.dtype == torch.bfloat16
        parity = parity_error(got, ref, bf16_out)
        parity_detail = {"err": parity, "bar": 2e-2 if w.dtype == "bf16" else 1e-4,
                         "raw_err": parity_error(got, ref, False), "tokens_per_sequence": Ts,
                         "sequences": w.B * w.H, "output": "bf16" if bf16_out else "f32",
                         "measure": "max|o - o_ref| / rms(o_ref)" + (" beyond each element's bf16 half-ulp"
                                                                     if bf16_out else "")}
    plan.close()

    if rank == 0:
        line = {
            "metric": NONLINEAR_METRIC if nonlinear else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": warm,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, **{k: getattr(w, k) for k in ("B", "H", "T", "dk", "dv", "L")},
                       "io": w.dtype, "l2": L2Flush.DESCRIPTION,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roofline, "path_roofline": path_roofline,
            # the goal is half of the binding resource's roofline at the 16K shape: how far the
            # dominant kernel and the whole forward are from it (x faster needed)
            "roofline_target": {"frac": ROOFLINE_TARGET, "kernel_gap": ROOFLINE_TARGET / roofline["frac"],
                                "path_gap": ROOFLINE_TARGET / path_roofline["frac"]},
            "kernels": kernels,
            "parity": parity, "parity_detail": parity_detail,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
            "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms),
            "graph_ms_per_step": graph_ms, "warm_l2_ms_per_step": warm_ms,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------------------------------------
DECODE_METRIC = "PRISM decode step tokens/s (one token per sequence, all heads) + % of HBM roofline"
TOKEN_KEYS = ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta")


def decode_alg_bytes(w):
    """Bytes one decode step must move: the fp32 state read and written once per (sequence,
    head), the token's inputs, the convolution history read and written, the output, and the
    convolution weights once."""
    io = 2 if w.dtype == "bf16" else 4
    per_head = (2 * w.dv * w.dk * 4 + io * (2 * w.dk + w.dv + w.R * w.dk) + 4 * (2 + 2 * w.R)
                + 2 * 3 * w.dv * io + w.dv * io)
    return w.B * w.H * per_head + w.H * 4 * w.dv * io


def decode_inputs(w, seed=0):
    import torch
    from ssm_sequence_layer_gb300.inputs import make_inputs
    inp = make_inputs(w.B, w.H, 1, w.dk, w.dv, w.L, dtype=w.dtype, seed=seed)
    tok = {k: (v[:, :, 0].contiguous() if k in TOKEN_KEYS else v) for k, v in inp.items()}
    g = torch.Generator().manual_seed(seed + 1)
    S = torch.randn(w.B, w.H, w.dv, w.dk, generator=g) * 0.3
    hist = torch.randn(w.B, w.H, 3, w.dv, generator=g).to(tok["v"].dtype)
    return inp, tok, S, hist


def decode_oracle_sample(w, inp, S, hist, seconds_target, nthreads, reps=None):
    """The oracle's step (T = 1 from S_init and v_hist) over all B*H heads, repeated for about
    `seconds_target` seconds (or `reps` times).  Returns (tokens/s, repetitions, seconds)."""
    from oracle import prism_oracle
    a = {k: (v.double().numpy() if hasattr(v, "double") else v) for k, v in inp.items()}
    S64, h64 = S.double().numpy(), hist.double().numpy()

    def once():
        prism_oracle.forward(a["q"], a["k"], a["v"], a["beta"], a["alpha"], a["u"], a["gamma"], a["eta"],
                             a["conv_w"], a["L"], S_init=S64, v_hist=h64, want_state=True, nthreads=nthreads)

    if reps is None:
        t0 = time.perf_counter()
        once()
        dt1 = time.perf_counter() - t0
        reps = max(1, int(seconds_target / max(dt1, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        once()
    dt = time.perf_counter() - t0
    return w.B * reps / dt, reps, dt


def run_decode(args, w):
    import torch

    from ssm_sequence_layer_gb300 import binding as Bd
    from ssm_sequence_layer_gb300 import build as cuda_build

    world, rank, local = dist_setup(args)
    if rank == 0:
        cuda_build.build()
    barrier(world)
    steps, warm = args.steps, max(args.warmup, 3)
    inp_cpu, tok_cpu, S_cpu, hist_cpu = decode_inputs(w)
    tok = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in tok_cpu.items()}
    S, hist = S_cpu.cuda(), hist_cpu.cuda()
    out = torch.empty(w.B, w.H, w.dv, dtype=tok["v"].dtype, device="cuda")
    stream = torch.cuda.current_stream()
    plan = Bd.Plan(w.B, w.H, 1, w.dk, w.dv, w.L, io=w.dtype)
    flush = L2Flush()
    for _ in range(warm):
        flush()
        plan.decode_step(tok, hist, S, out, stream)
    torch.cuda.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):  # one kernel per step: the step events time the decode kernel itself
        flush()
        ev[i][0].record(stream)
        plan.decode_step(tok, hist, S, out, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    plan.last_device_status()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = sum(step_ms) / steps
    ms = max_over_ranks(ms_local, world)
    value = w.B * world / (ms / 1e3)
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    alg = decode_alg_bytes(w)
    achieved = alg / (ms_local / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "decode", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic_from_profiles("decode", w.name),
                "alg_bytes_per_launch": alg, "kernel_ms": ms_local, "peak_source": f"{peak_kind} hbm_gbs"}

    e2e = None
    if not args.no_e2e:  # the token's inputs from pinned host memory, the output back; the state stays resident
        host = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in tok_cpu.items()}
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for k, v in host.items() if torch.is_tensor(v) and k != "conv_w"
                  and (w.L > 1 or k not in ("u", "gamma", "eta")))
        dtok = {k: (torch.empty_like(v, device="cuda") if torch.is_tensor(v) else v) for k, v in host.items()}
        e2e_ms = []
        for i in range(max(3, min(steps, 20)) + 2):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k, v in host.items():
                if torch.is_tensor(v) and k != "conv_w":
                    dtok[k].copy_(v, non_blocking=True)
            plan.decode_step(dtok, hist, S, out, stream)
            hout.copy_(out, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                e2e_ms.append(a.elapsed_time(b))
        e2e_ms_mean = max_over_ranks(sum(e2e_ms) / len(e2e_ms), world)
        e2e = {"value": w.B * world / (e2e_ms_mean / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": hout.numel() * hout.element_size(), "ms_per_step": e2e_ms_mean}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = max(1, min(len(os.sched_getaffinity(0)), w.B * w.H))
        v, reps, dt = decode_oracle_sample(w, inp_cpu, S_cpu, hist_cpu, args.cpu_seconds, nthreads)
        cpu = {"value": v, "unit": UNIT, **host_info(nthreads), "kind": "oracle",
               "sample": f"fp64 oracle, one token for all {w.B * w.H} (sequence, head) pairs, {reps} times ({dt:.1f} s)"}
    plan.close()
    if rank == 0:
        line = {
            "metric": DECODE_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, **{k: getattr(w, k) for k in ("B", "H", "dk", "dv", "L")},
                       "io": w.dtype, "state": "fp32, resident", "l2": L2Flush.DESCRIPTION,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": steps, "clocks": clocks,
            "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


PROJECT_METRIC = "PRISM input projections tokens/s (ShortConv + basis/gain/gate GEMM) + % of roofline"


def run_project(args, name):
    import torch

    from ssm_sequence_layer_gb300 import binding as Bd
    from ssm_sequence_layer_gb300 import build as cuda_build
    from ssm_sequence_layer_gb300.inputs import PROJECTION_WORKLOADS, make_projection_inputs

    world, rank, local = dist_setup(args)
    if rank == 0:
        cuda_build.build()
    barrier(world)
    cfg = PROJECTION_WORKLOADS[name]
    B_, T, D, H, R, dk, dv = (cfg[k] for k in ("B", "T", "D", "H", "R", "dk", "dv"))
    N = H * R * (dk + dv + 1)
    steps, warm = args.steps, max(args.warmup, 3)
    pi = make_projection_inputs(B_, T, D, H, R, dk, dv, seed=0)
    X, cw, W = pi["X"].cuda(), pi["conv_x"].cuda(), pi["W"].cuda()
    plan = Bd.Plan(B_, H, T, dk, dv, R + 1, io="bf16")
    out = (torch.empty(B_, H, T, R, dk, dtype=torch.bfloat16, device="cuda"),
           torch.empty(B_, H, T, R, dv, dtype=torch.bfloat16, device="cuda"),
           torch.empty(B_, H, T, R, dtype=torch.float32, device="cuda"))
    stream = torch.cuda.current_stream()
    flush = L2Flush()
    for _ in range(warm):
        flush()
        plan.project(X, cw, W, out, stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        plan.project(X, cw, W, out, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    plan.last_device_status()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = sum(step_ms) / steps
    ms = max_over_ranks(ms_local, world)
    tokens = B_ * T
    value = tokens * world / (ms / 1e3)
    peaks, peak_kind = load_peaks()
    flops = 2.0 * tokens * D * N
    alg_bytes = 2 * tokens * D + 2 * N * D + 8 * D + tokens * H * R * (2 * dk + 2 * dv + 4)
    t_hbm = alg_bytes / (float(peaks["hbm_gbs"]) * 1e9)
    t_tc = flops / (float(peaks["bf16_tflops"]) * 1e12)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    if bound == "tensor":
        ach = flops / (ms_local / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": float(peaks["bf16_tflops"]), "unit": "TFLOP/s",
                "frac": ach / float(peaks["bf16_tflops"]), "peak_source": f"{peak_kind} bf16_tflops"}
    else:
        ach = alg_bytes / (ms_local / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": ach / float(peaks["hbm_gbs"]), "peak_source": f"{peak_kind} hbm_gbs"}
    roof.update(kernel="project", traffic=traffic_from_profiles("project", name), alg_bytes_per_launch=alg_bytes,
                alg_flops_per_launch=flops, kernel_ms=ms_local,
                hbm_frac=alg_bytes / (ms_local / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
                tensor_frac=flops / (ms_local / 1e3) / 1e12 / float(peaks["bf16_tflops"]))
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import prism_projection
        Ts = min(T, 512)
        sub = pi["X"][:, :Ts]
        t0 = time.perf_counter()
        prism_projection.project(sub, pi["conv_x"], pi["W"], H, R, dk, dv)
        dt = time.perf_counter() - t0
        cpu = {"value": B_ * Ts / dt, "unit": UNIT, **host_info(len(os.sched_getaffinity(0))), "kind": "oracle",
               "sample": f"numpy fp64 oracle over the first {Ts} tokens of all {B_} sequences ({dt:.2f} s)"}
    plan.close()
    if rank == 0:
        line = {
            "metric": PROJECT_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": name, **cfg, "N": N, "l2": L2Flush.DESCRIPTION,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": None, "gpu_launches": steps, "clocks": clocks,
            "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


BACKWARD_METRIC = "PRISM layer bwd tokens/s (all input cotangents, T=16K) + % of HBM roofline"
BWD_KEYS = ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta", "conv_w")


def backward_kernel_bytes(name, w, nl=False):
    """Bytes a backward kernel must move at minimum for one launch over the workload: each of
    its inputs read once and each of its outputs written once, the intermediates of the design
    included (token-serial form: the per-token states S_{t-1} and cotangents dS_t, fp32, dv dk
    floats per token each; chunked form: four fp32 chunk maps, the chunk states and cotangents,
    and the fp16 stash of 5 + R tiles per chunk).  With ``nl`` (the non-linear chain) the gains p
    [R dv] per token, in the io dtype, take the place of eta, and dp (fp32) that of deta."""
    io = 2 if w.dtype == "bf16" else 4
    th = w.B * w.H * w.T
    R = w.R
    qk = th * w.dk * io
    v = th * w.dv * io
    u = th * R * w.dk * io
    gates2 = th * 8
    X = dX = th * R * w.dv * 4
    state = th * w.dv * w.dk * 4
    per_row = th * w.dv * 4  # z, dout, dh or a dv-sized fp32 cotangent
    ntile = -(-w.T // 64)
    chunks = w.B * w.H * ntile
    dd = w.dk * w.dv * 4
    tile = 64 * w.dv * 2
    gates = th * 4 * (2 + (1 if nl else 2) * R)
    pg = th * R * w.dv * io if nl else 0    # the gains read
    dpg = th * R * w.dv * 4 if nl else 0    # their cotangent written
    eta_rw = 0 if nl else th * 4 * R        # eta read or deta written
    table = {
        "bwd_maps": 2 * qk + v + u + gates + pg + per_row + 4 * chunks * dd + chunks * (5 + R) * tile,
        "bwd_chunk_scan": 4 * chunks * dd + (2 * chunks + w.B * w.H) * dd,
        # the chunk's inputs, dout, S_c, S_{c+1}, G_c, the stash read; dv, dX, dbeta, dq, dk, du, dalpha written
        "bwd_grad": 2 * qk + v + u + gates + per_row + 3 * chunks * dd + chunks * (5 + R) * tile
        + per_row + dX + th * 4 + 2 * th * w.dk * 4 + th * R * w.dk * 4 + th * 4,
        "bwd_factors": v + th * 4 * R + eta_rw + pg + X,
        # both halves of the scan launch: S_{t-1} forward, dS_t (with z, dx) in reverse
        "bwd_scan": (qk + v + u + gates2 + X + state) + (2 * qk + u + gates2 + per_row + state + per_row + dX),
        "bwd_token_grad": 2 * qk + v + u + gates2 + X + 2 * state + 2 * per_row + 2 * th * w.dk * 4 + per_row
        + th * R * w.dk * 4 + th * 8,
        "bwd_chain_grad": v + th * 4 * R + eta_rw + pg + dX + 2 * per_row + per_row + th * 4 * R + eta_rw + dpg,
        "bwd_conv_grad": v + 3 * per_row + w.B * w.H * ntile * 4 * w.dv * 4,
        # the fused tail (bf16, dv = 64): the chain's reads and dv once read and once written; dH stays on chip
        "bwd_tail": v + th * 4 * R + eta_rw + pg + dX + 2 * per_row + th * 4 * R + eta_rw + dpg
        + w.B * w.H * ntile * 4 * w.dv * 4,
        "bwd_conv_reduce": w.B * w.H * ntile * 4 * w.dv * 4 + w.H * 4 * w.dv * 4,
    }
    return table[name]


def backward_path_bytes(w, nl=False):
    """The pass's own minimum: the inputs and dout read once, every cotangent written once (with
    ``nl``, the gains p and their cotangent in place of eta and deta)."""
    io = 2 if w.dtype == "bf16" else 4
    th = w.B * w.H * w.T
    R = w.R
    ins = th * (2 * w.dk + w.dv + R * w.dk) * io + th * 4 * (2 + 2 * R) + th * w.dv * 4
    outs = th * 4 * (2 * w.dk + w.dv + 2 + R * w.dk + 2 * R)
    if nl:
        ins += th * R * w.dv * io - th * 4 * R
        outs += th * R * w.dv * 4 - th * 4 * R
    return ins + outs


def backward_oracle_step(sub, dout, nthreads):
    from oracle import prism_backward
    prism_backward.backward(sub["q"], sub["k"], sub["v"], sub["beta"], sub["alpha"], sub["u"], sub["gamma"],
                            sub["eta"], sub["conv_w"], sub["L"], dout, p_gain=sub.get("p_gain"), nthreads=nthreads)


def backward_sample(inp, dout, Ts):
    sub = {k: (v[:, :, :Ts].contiguous() if hasattr(v, "shape") and k != "conv_w" else v) for k, v in inp.items()}
    sub = {k: (v.double().numpy() if hasattr(v, "double") else v) for k, v in sub.items()}
    return sub, dout[:, :, :Ts].double().numpy()


def run_backward(args, w):
    import torch

    from ssm_sequence_layer_gb300 import binding as Bd
    from ssm_sequence_layer_gb300 import build as cuda_build
    from ssm_sequence_layer_gb300.inputs import make_cotangents, make_gain, make_workload_inputs

    world, rank, local = dist_setup(args)
    if rank == 0:
        cuda_build.build()
    barrier(world)
    steps, warm = args.steps, max(args.warmup, 3)
    nl = args.nonlinear and w.L > 1
    inp_cpu = make_workload_inputs(w, seed=0)
    if nl:  # the non-linear residual chain: gains p in place of eta
        inp_cpu["p_gain"] = make_gain(w.B, w.H, w.T, w.L, w.dv, dtype=w.dtype, seed=0)
    dout_cpu, _ = make_cotangents(w.B, w.H, w.T, w.dk, w.dv, seed=0)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp_cpu.items()}
    dout = dout_cpu.cuda()
    stream = torch.cuda.current_stream()
    plan = Bd.Plan.for_inputs(dev, path=args.path or None)  # --path 1: the token-serial form
    flush = L2Flush()

    def step(d, dz, g=None):
        return plan.backward(d, dz, grads=g, stream=stream, p_gain=d["p_gain"] if nl else None)

    grads = step(dev, dout)
    for _ in range(warm):
        flush()
        step(dev, dout, grads)
    torch.cuda.synchronize()
    plan.last_device_status()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        step(dev, dout, grads)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    plan.last_device_status()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    plan.set_option(Bd.PRISM_OPT_TIMING, 1)
    per_kernel, launches = {}, 0
    for _ in range(steps):
        flush()
        step(dev, dout, grads)
        torch.cuda.synchronize()
        kt = plan.kernel_times()
        launches += len(kt)
        for name, ms in kt:
            per_kernel.setdefault(name, []).append(ms)
    plan.set_option(Bd.PRISM_OPT_TIMING, 0)
    plan.last_device_status()
    ms_local = sum(step_ms) / steps
    ms = max_over_ranks(ms_local, world)
    tokens = w.B * w.T
    value = tokens * world / (ms / 1e3)
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tot = {n: sum(v) for n, v in per_kernel.items()}
    dom = max(tot, key=tot.get)
    dom_ms = tot[dom] / len(per_kernel[dom])
    dom_bytes = backward_kernel_bytes(dom, w, nl)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic_from_profiles(dom, w.name + ("_nonlinear" if nl else "")),
                "alg_bytes_per_launch": dom_bytes, "kernel_ms": dom_ms, "peak_source": f"{peak_kind} hbm_gbs"}
    kernels = {n: {"ms_mean": tot[n] / len(per_kernel[n]), "share": tot[n] / sum(tot.values()),
                   "hbm_frac": backward_kernel_bytes(n, w, nl) / (tot[n] / len(per_kernel[n]) / 1e3) / 1e9 / hbm}
               for n in tot}
    pb = backward_path_bytes(w, nl)
    path_roofline = {"achieved": pb / (ms_local / 1e3) / 1e9, "unit": "GB/s",
                     "frac": pb / (ms_local / 1e3) / 1e9 / hbm, "alg_bytes_per_step": pb}

    e2e = None
    if not args.no_e2e:  # inputs and dout copied in from pinned host memory, every cotangent copied back
        host = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in inp_cpu.items()}
        hdout = dout_cpu.pin_memory()
        hgrads = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in grads.items()}
        used = [k for k in BWD_KEYS + (("p_gain",) if nl else ())
                if (w.L > 1 or k not in ("u", "gamma", "eta")) and not (nl and k == "eta")]
        h2d = hdout.numel() * 4 + sum(host[k].numel() * host[k].element_size() for k in used)
        d2h = sum(v.numel() * v.element_size() for k, v in hgrads.items()
                  if w.L > 1 or k not in ("du", "dgamma", "deta"))
        dbuf = {k: (torch.empty_like(v, device="cuda") if torch.is_tensor(v) else v) for k, v in host.items()}
        ddout = torch.empty_like(hdout, device="cuda")
        e2e_ms = []
        for i in range(max(3, min(steps, 10)) + 2):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k in used:
                dbuf[k].copy_(host[k], non_blocking=True)
            ddout.copy_(hdout, non_blocking=True)
            step(dbuf, ddout, grads)
            for k, v in hgrads.items():
                v.copy_(grads[k], non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                e2e_ms.append(a.elapsed_time(b))
        e2e_mean = max_over_ranks(sum(e2e_ms) / len(e2e_ms), world)
        e2e = {"value": tokens * world / (e2e_mean / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_mean}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = cpu_threads(w)
        Ts = min(w.T, 256)
        sub, sd = backward_sample(inp_cpu, dout_cpu, Ts)
        t0 = time.perf_counter()
        backward_oracle_step(sub, sd, nthreads)
        dt = time.perf_counter() - t0
        Ts = int(min(w.T, max(Ts, Ts * args.cpu_seconds / max(dt, 1e-3))))
        sub, sd = backward_sample(inp_cpu, dout_cpu, Ts)
        t0 = time.perf_counter()
        backward_oracle_step(sub, sd, nthreads)
        dt = time.perf_counter() - t0
        cpu = {"value": w.B * Ts / dt, "unit": UNIT, **host_info(nthreads), "kind": "oracle",
               "sample": f"fp64 backward oracle over the first {Ts} tokens of all {w.B * w.H} sequences ({dt:.1f} s)"}
    plan.close()
    if rank == 0:
        chunked = "bwd_maps" in per_kernel  # which form the library took (the kernels it launched)
        line = {
            "metric": BACKWARD_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            # the chunked form's products take fp16 operands (fp32 accumulation); the token-serial form is fp32
            "dtype": "f16" if chunked else "f32", "data": "synthetic",
            "config": {"workload": w.name, **{k: getattr(w, k) for k in ("B", "H", "T", "dk", "dv", "L")},
                       "io": w.dtype, "form": "chunked" if chunked else "token-serial",
                       "chain": "non-linear" if nl else "linear", "l2": L2Flush.DESCRIPTION,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roofline, "path_roofline": path_roofline, "kernels": kernels, "cpu_baseline": cpu,
            "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
            "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_backward_reference(args, w):
    """The backward oracle as the reference arm: each step is the oracle's backward over the
    first Ts tokens of every sequence of the workload, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    world = int(os.environ.get("WORLD_SIZE", "1"))
    from ssm_sequence_layer_gb300.inputs import make_cotangents, make_workload_inputs
    inp = make_workload_inputs(w)
    dout, _ = make_cotangents(w.B, w.H, w.T, w.dk, w.dv, seed=0)
    nthreads = cpu_threads(w)
    Ts = min(w.T, 512)
    sub, sd = backward_sample(inp, dout, Ts)
    for _ in range(max(args.warmup, 0)):
        backward_oracle_step(sub, sd, nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        backward_oracle_step(sub, sd, nthreads)
    dt = time.perf_counter() - t0
    value = w.B * Ts * args.steps / dt
    line = {
        "impl": "reference", "metric": BACKWARD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **{k: getattr(w, k) for k in ("B", "H", "T", "dk", "dv", "L")}, "io": w.dtype},
        "cpu_baseline": {"value": value, "unit": UNIT, **host_info(nthreads), "kind": "oracle",
                         "sample": f"backward oracle over the first {Ts} tokens of all {w.B * w.H} sequences per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    from ssm_sequence_layer_gb300.inputs import DECODE_WORKLOADS, WORKLOADS
    if args.mode == "decode":
        w = DECODE_WORKLOADS[args.workload or "decode_lm130m"]
        if args.impl == "reference":
            return run_decode_reference(args, w)
        return run_decode(args, w)
    if args.mode == "project":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm covers the forward and the decode step"}))
            return 0
        return run_project(args, args.workload or "project_lm130m")
    if args.mode == "backward":
        w = WORKLOADS[args.workload or "seqrec_16k"]
        if args.seq_len:
            w = dataclasses.replace(w, T=args.seq_len, name=f"{w.name}_T{args.seq_len}")
        if args.impl == "reference":
            return run_backward_reference(args, w)
        return run_backward(args, w)
    if args.mode == "nonlinear":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm covers the forward and the decode step"}))
            return 0
        w = WORKLOADS[args.workload or "lm130m_layer"]
        if args.seq_len:
            w = dataclasses.replace(w, T=args.seq_len, name=f"{w.name}_T{args.seq_len}")
        return run_ours(args, w)
    w = WORKLOADS[args.workload or "seqrec_16k"]
    if args.seq_len:
        w = dataclasses.replace(w, T=args.seq_len, name=f"{w.name}_T{args.seq_len}")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


def run_decode_reference(args, w):
    """The oracle as the reference arm of the decode step: each step is the oracle's step over
    all (sequence, head) pairs on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    world = int(os.environ.get("WORLD_SIZE", "1"))
    inp, _, S, hist = decode_inputs(w)
    nthreads = max(1, min(len(os.sched_getaffinity(0)), w.B * w.H))
    if args.warmup > 0:
        decode_oracle_sample(w, inp, S, hist, 0.0, nthreads, reps=args.warmup)
    _, _, dt = decode_oracle_sample(w, inp, S, hist, 0.0, nthreads, reps=args.steps)
    value = w.B * args.steps / dt
    line = {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **{k: getattr(w, k) for k in ("B", "H", "dk", "dv", "L")}, "io": w.dtype},
        "cpu_baseline": {"value": value, "unit": UNIT, **host_info(nthreads), "kind": "oracle",
                         "sample": f"oracle step over all {w.B * w.H} (sequence, head) pairs"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
