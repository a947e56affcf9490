#!/usr/bin/env python
"""Benchmark of the fused weight-gradient + AdamW step (libforge) on GB300.

One step = one fused forge_wgrad_adamw call on each of the seven projections
of a Llama-3.1-8B decoder layer (q, k, v, o, gate, up, down) at a fixed token
count, inputs resident in HBM.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle arm

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas: the path has no cross-rank exchange), the timed region
is bracketed by barriers, and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import glob
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from weight_gradient_gemm_gb300.inputs import (LLAMA31_8B_SHAPES, bf16_bits,  # noqa: E402
                                               make_step_inputs)

METRIC = "fused wgrad+AdamW TFLOP/s and % roofline, Llama-3.1-8B linears, 1 GB300"
HYPER = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
# the other optimizers, with the FORGE page's shared settings per family (its
# appendix table of optimizer families: lr, wd, betas, eps; momentum 0.9)
_FAM = dict(lr=2e-5, weight_decay=1e-2)
OPT_HYPER = [dict(_FAM), dict(_FAM, momentum=0.9), dict(_FAM, eps=1e-10), dict(_FAM, eps=1e-8),
             dict(lr=3e-6, weight_decay=1.0, beta1=0.9, beta2=0.99),
             dict(_FAM, beta1=0.9, beta2=0.999, eps=1e-8),
             dict(_FAM, beta1=0.9, beta2=0.999, eps=1e-8)]
FMT_NAMES = {0: "fp32", 1: "bf16", 2: "int8_block128", 3: "fp8_e4m3_per_tensor"}
# bytes per parameter: W read + write, m and v read + write (+ int8 block
# scales; fp8's 16 bytes per tensor are not counted)
STATE_BYTES = {0: 20.0, 1: 12.0, 2: 8.0 + 16.0 / 128.0, 3: 8.0}
FP8_HEADROOM = 2.0
L2_BYTES = 126 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOADS = {
    # name: (config index of the recipe, BT, moment format, dY std, spike fraction)
    "llama31_8b_layer_bt512_fp32": (1, 512, 0, 1e-3, 0.0),
    "llama31_8b_layer_bt512_bf16": (2, 512, 1, 1e-3, 0.01),
    "llama31_8b_layer_bt2048_bf16": (2, 2048, 1, 1e-3, 0.01),
    "llama31_8b_layer_bt8192_bf16": (2, 8192, 1, 1e-3, 0.01),
    "llama31_8b_layer_bt4096_int8": (3, 4096, 2, 1e-3, 0.0),
    "llama31_8b_layer_bt512_fp8": (4, 512, 3, 1e-3, 0.0),
}
DEFAULT_WORKLOAD = "llama31_8b_layer_bt512_fp32"
_RECIPE = {"fp32": (1, 0, 1e-3, 0.0), "bf16": (2, 1, 1e-3, 0.01), "int8": (3, 2, 1e-3, 0.0),
           "fp8": (4, 3, 1e-3, 0.0)}


def workload_spec(name: str):
    """(recipe config, BT, moment format, dY std, spike fraction) of a named
    workload; besides the table, any llama31_8b_layer_bt<BT>_<fp32|bf16|int8|fp8>."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    parts = name.split("_")
    if len(parts) == 5 and name.startswith("llama31_8b_layer_bt") and parts[4] in _RECIPE:
        cfg, fmt, dy_std, spike = _RECIPE[parts[4]]
        return (cfg, int(parts[3][2:]), fmt, dy_std, spike)
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest() -> str:
    """Hash of the kernel sources; a stored ncu traffic figure is used only
    while it matches."""
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "weight_gradient_gemm_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str):
    """ncu DRAM bytes per launch of the fused kernel for this workload, from
    profiles/, if the profile was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"forge_gemm_fused_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_sha256") != source_digest():
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = None
        if not inside:   # timed window shorter than the sampling period
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
            note = "nearest sample (window shorter than 100 ms)"
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in inside for n, v in zip(names, p[5:9]) if v.lower() == "active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
               "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

class Layer:
    """Device buffers of one decoder layer's seven projections."""

    def __init__(self, cfg, bt, fmt, dy_std, spike, dev, with_host=True, only=None):
        from weight_gradient_gemm_gb300 import forge as F
        self.items = []
        # fp8 moments: every tensor's scale record in one buffer, rolled after each step
        self.fp8_scales = F.alloc_fp8_scales(14, device=dev) if fmt == 3 else None
        for i, (name, d_out, d_in) in enumerate(LLAMA31_8B_SHAPES):
            if only and name not in only:
                continue
            s = make_step_inputs(cfg, i, 0, bt, d_in, d_out, x_std=1.0, dy_std=dy_std,
                                 with_w=True, spike_frac=spike)
            x_host = s.x.pin_memory() if with_host else None
            dy_host = s.dy.pin_memory() if with_host else None
            m, v, ms, vs = F.alloc_moments(d_out, d_in, fmt, dev)
            if fmt == 3:
                ms, vs = self.fp8_scales[2 * i], self.fp8_scales[2 * i + 1]
            self.items.append(dict(
                name=name, d_in=d_in, d_out=d_out, x=s.x.to(dev), dy=s.dy.to(dev),
                w=s.w.to(dev), m=m, v=v, ms=ms, vs=vs, x_host=x_host, dy_host=dy_host))
        self.bt = bt
        self.fmt = fmt
        # q, k, v read the same activations X in the model; here each projection
        # has its own seeded X (the work per step is the same)
        self.group = [dict(X=it["x"], dY=it["dy"], W=it["w"], m=it["m"], v=it["v"],
                           m_scale=it["ms"], v_scale=it["vs"]) for it in self.items]

    def second_input_set(self):
        """The same layers with their own device X and dY buffers (for inputs
        staged while the previous step computes)."""
        return [dict(g, X=torch.empty_like(g["X"]), dY=torch.empty_like(g["dY"]))
                for g in self.group]

    def flops(self):
        return sum(2.0 * self.bt * it["d_in"] * it["d_out"] for it in self.items)

    def params(self):
        return sum(it["d_in"] * it["d_out"] for it in self.items)

    def alg_bytes(self):
        return sum(it["d_in"] * it["d_out"] * STATE_BYTES[self.fmt]
                   + 2.0 * self.bt * (it["d_in"] + it["d_out"]) for it in self.items)

    def h2d_bytes(self):
        return sum(2 * self.bt * (it["d_in"] + it["d_out"]) for it in self.items)


def fused_step(F, layer, step, events=None, stream=None):
    """One step: the seven projections in one grouped launch (with fp8
    moments, then the scale roll of delayed scaling)."""
    if events is not None:
        events[0][0].record(stream)
    F.wgrad_adamw_grouped(layer.group, step=step, **HYPER)
    if layer.fp8_scales is not None:
        F.fp8_roll_scales(layer.fp8_scales, FP8_HEADROOM)
    if events is not None:
        events[0][1].record(stream)


def fused_step_separate(F, layer, step, events=None, stream=None):
    """The same step as seven separate launches (one per projection)."""
    for i, it in enumerate(layer.items):
        if events is not None:
            events[i][0].record(stream)
        F.wgrad_adamw(it["x"], it["dy"], it["w"], it["m"], it["v"], step=step,
                      m_scale=it["ms"], v_scale=it["vs"], **HYPER)
        if events is not None:
            events[i][1].record(stream)


def max_over_ranks(values, dev):
    """Each value's maximum over the ranks of the process group (the slowest
    replica sets the job's time).  `dev` is where the reduction runs: the
    rank's GPU under NCCL, the CPU under gloo."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_value(world, units_per_rank, seconds):
    """Whole-job throughput of `world` replicas that each process
    `units_per_rank` in `seconds` (the maximum over ranks)."""
    return world * units_per_rank / seconds


def run_gpu(args, rank, world, dev):
    from weight_gradient_gemm_gb300 import forge as F
    F.lib()
    cfg, bt, fmt, dy_std, spike = workload_spec(args.workload)
    layer = Layer(cfg, bt, fmt, dy_std, spike, dev,
                  only=args.only.split(",") if args.only else None)
    stream = torch.cuda.current_stream()
    dist = world > 1

    def barrier():
        if dist:
            torch.distributed.barrier()

    # moments warmed by 10 prior steps (same seeded inputs), then W warm-up steps
    step = 0
    for _ in range(10):
        step += 1
        fused_step(F, layer, step)
    for _ in range(args.warmup):
        step += 1
        fused_step(F, layer, step)
    assert F.device_error() == 0

    # ---- timed region: K steps, each one grouped launch timed on the launch stream
    n = len(layer.items)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))]
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.25 if sampler else 0.0)
    barrier()
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    t_start.record(stream)
    for k in range(args.steps):
        step += 1
        fused_step(F, layer, step, ev[k], stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    barrier()
    status = F.device_error()
    if status != 0:
        raise RuntimeError(F.status_string(status))
    elapsed_ms = t_start.elapsed_time(t_end)
    launch_ms = [a.elapsed_time(b) for row in ev for (a, b) in row]
    kern_ms = sum(launch_ms)
    if dist:
        elapsed_ms, kern_ms = max_over_ranks([elapsed_ms, kern_ms], dev)

    # ---- the same launch repeated for about a second (diagnostic, after the
    # timed region): per-launch statistics over a window long enough for the
    # clock sampler, with the clock samples binned by quarter of the window
    steady = None
    if rank == 0 and not args.no_diagnostics:
        est = max(kern_ms / max(1, args.steps), 1e-3)
        n_st = int(min(20000, max(args.steps, math.ceil(1000.0 / est))))
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_st)]
        torch.cuda.synchronize()
        s0 = time.perf_counter()
        for k in range(n_st):
            step += 1
            fused_step(F, layer, step, [sev[k]], stream)
        torch.cuda.synchronize()
        s1 = time.perf_counter()
        steady = dict(launch_ms=[a.elapsed_time(b) for a, b in sev], w0=s0, w1=s1)
    if sampler:
        sampler.stop()

    if args.no_diagnostics:
        return dict(layer=layer, elapsed_ms=elapsed_ms, kern_ms=kern_ms, launch_ms=launch_ms,
                    steady=None, sampler=sampler, unf_ms=None, per_proj_ms=None, backward=None,
                    opt_ms=None, opt_fmt=None, acc_ms=None, sr_ms=None, e2e=None, e2e_ms=None,
                    clocks=sampler.summary(w0, w1) if sampler else None,
                    config=F.describe_config(bt, 4096, 4096, fmt))

    # ---- diagnostics (not the reported value): the same step as seven launches
    sep_steps = max(3, min(args.steps, 30))
    sev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)] for _ in range(sep_steps)]
    for k in range(sep_steps):
        step += 1
        fused_step_separate(F, layer, step, sev[k], stream)
    torch.cuda.synchronize()
    per_proj_ms = [sum(row[i][0].elapsed_time(row[i][1]) for row in sev) / sep_steps
                   for i in range(n)]

    # ---- unfused comparison arm: forge_wgrad (bf16 dW) + forge_adamw
    unf_steps = max(3, min(args.steps, 50))
    dw = torch.empty(max(it["d_in"] * it["d_out"] for it in layer.items), dtype=torch.bfloat16,
                     device=dev)
    for _ in range(2):
        step += 1
        unfused_step(F, layer, step, dw)
    barrier()
    torch.cuda.synchronize()
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    u0.record(stream)
    for _ in range(unf_steps):
        step += 1
        unfused_step(F, layer, step, dw)
    u1.record(stream)
    torch.cuda.synchronize()
    unf_ms = u0.elapsed_time(u1) / unf_steps
    assert F.device_error() == 0

    # ---- the layer's whole backward step (diagnostic, not the reported
    # value): forge_linear_backward per projection (dX = dY W from the weight
    # before the update, then the fused step), dX alone (forge_dgrad), and
    # cuBLAS's dX (torch.matmul) on the same tensors for scale
    bw_steps = max(3, min(args.steps, 30))
    dx = [torch.empty((bt, it["d_in"]), dtype=torch.bfloat16, device=dev) for it in layer.items]

    def per_step_ms(fn):
        fn()
        torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(bw_steps):
            fn()
        b1.record(stream)
        torch.cuda.synchronize()
        return b0.elapsed_time(b1) / bw_steps

    dg_items = [dict(dY=it["dy"], W=it["w"], dX=o) for it, o in zip(layer.items, dx)]
    ws_bytes = F.dgrad_workspace_bytes(dg_items)
    dws = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=dev) if ws_bytes else None

    def dgrad_all():
        F.dgrad_grouped(dg_items, workspace=dws)

    def dgrad_each():
        for it, o in zip(layer.items, dx):
            F.dgrad(it["dy"], it["w"], o)

    def cublas_dgrad_all():
        for it, o in zip(layer.items, dx):
            torch.matmul(it["dy"], it["w"], out=o)

    bw_layers = [dict(g, dX=o) for g, o in zip(layer.group, dx)]

    def backward_all():
        nonlocal step
        step += 1
        F.linear_backward_grouped(bw_layers, step=step, workspace=dws, **HYPER)

    # ---- the other optimizers (diagnostic): forge_wgrad_opt_grouped over the
    # layer (one launch), states in the workload's format (fp32 for 8-bit
    # workloads), zeroed first
    sfmt = fmt if fmt in (F.MOM_FP32, F.MOM_BF16) else F.MOM_FP32
    sdt = torch.float32 if sfmt == F.MOM_FP32 else torch.bfloat16
    sbuf = [[torch.zeros((it["d_out"], it["d_in"]), dtype=sdt, device=dev) for _ in range(2)]
            for it in layer.items]
    opt_ms = {}
    for opt in range(7):
        for pair in sbuf:
            for b in pair:
                b.zero_()
        n_st = F.OPT_STATES[opt]
        ost = [0]
        olayers = [dict(X=it["x"], dY=it["dy"], W=it["w"],
                        s1=pair[0] if n_st >= 1 else None, s2=pair[1] if n_st >= 2 else None)
                   for it, pair in zip(layer.items, sbuf)]

        def opt_step():
            ost[0] += 1
            F.wgrad_opt_grouped(olayers, opt, step=ost[0], **OPT_HYPER[opt])
        opt_ms[opt] = per_step_ms(opt_step)
    assert F.device_error() == 0
    del sbuf, olayers

    # ---- the accumulate mode (diagnostic): forge_wgrad_accumulate_grouped
    # over the layer into fp32 buffers, with beta = 1 (B read and written) and
    # beta = 0 (B written only)
    acc_items = [dict(X=it["x"], dY=it["dy"],
                      B=torch.zeros((it["d_out"], it["d_in"]), dtype=torch.float32, device=dev))
                 for it in layer.items]

    def accumulate_all(beta):
        F.wgrad_accumulate_grouped(acc_items, beta)
    acc_ms = {b: per_step_ms(lambda b=b: accumulate_all(b)) for b in (1.0, 0.0)}
    # the step at the final micro-batch: AdamW on fp32(B + G) in one grouped
    # launch, against the last accumulate followed by forge_adamw on B
    if fmt in (F.MOM_FP32, F.MOM_BF16):
        final_layers = [dict(g, B=a["B"]) for g, a in zip(layer.group, acc_items)]

        def final_all():
            nonlocal step
            step += 1
            F.wgrad_adamw_acc_grouped(final_layers, step=step, **HYPER)

        def final_unfused():
            nonlocal step
            step += 1
            F.wgrad_accumulate_grouped(acc_items, 1.0)
            for g, a in zip(layer.group, acc_items):
                F.adamw(a["B"], g["W"], g["m"], g["v"], step=step, **HYPER)
        acc_ms["final"] = per_step_ms(final_all)
        acc_ms["final_unfused"] = per_step_ms(final_unfused)
        del final_layers
    assert F.device_error() == 0
    del acc_items

    # ---- the stochastic-rounding store (diagnostic): the fused step over the
    # layer in one launch with W committed by stochastic rounding (fp32 and
    # bf16 moments)
    sr_ms = None
    if fmt in (F.MOM_FP32, F.MOM_BF16):
        seeds = [1000 + k for k in range(len(layer.items))]

        def sr_all():
            nonlocal step
            step += 1
            F.wgrad_adamw_sr_grouped(layer.group, seeds, step=step, **HYPER)
        sr_ms = per_step_ms(sr_all)
        assert F.device_error() == 0

    backward = dict(dgrad_ms=per_step_ms(dgrad_all), dgrad_each_ms=per_step_ms(dgrad_each),
                    cublas_dgrad_ms=per_step_ms(cublas_dgrad_all),
                    linear_backward_ms=per_step_ms(backward_all), workspace_bytes=ws_bytes,
                    dgrad_config=F.describe_dgrad_config(bt, 4096, 14336))
    assert F.device_error() == 0

    # ---- end to end through the public API with host buffers: every step
    # copies its X and dY from pinned host memory, runs the grouped fused call
    # and reads back the library's status word (4 bytes).  As a training loop
    # would, the copies of step k+1 run on a second stream while step k
    # computes, into the other of two device input sets; step 0's copies are
    # inside the timed region too, and no step starts before its own inputs
    # have landed.
    e2e_steps = max(args.steps, 50)
    sets = [layer.group, layer.second_input_set()]
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]
    cp_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(e2e_steps)]
    st_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(e2e_steps)]

    def stage_inputs(b, k):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[b])      # the step that last read set b is done
            cp_ev[k][0].record(copy_stream)
            for it, g in zip(layer.items, sets[b]):
                g["X"].copy_(it["x_host"], non_blocking=True)
                g["dY"].copy_(it["dy_host"], non_blocking=True)
            cp_ev[k][1].record(copy_stream)
            copied[b].record(copy_stream)

    # the host-to-device bandwidth of the step's copies alone (pinned memory)
    h2d_ms = []
    for _ in range(5):
        stage_inputs(0, 0)
        torch.cuda.synchronize()
        h2d_ms.append(cp_ev[0][0].elapsed_time(cp_ev[0][1]))
    # each step's result read back: 4 bytes of the first projection's new W,
    # copied asynchronously into pinned memory after the step; the host reads
    # step k-1's while step k runs (a training loop's double-buffered readback),
    # and the library's status word is checked once at the end
    res_host = [torch.empty(2, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    res_ev = [torch.cuda.Event(), torch.cuda.Event()]
    w_first = layer.group[0]["W"].view(-1)
    checked = []
    # warm-up steps of the same loop (each input set used once: its tensor
    # maps encoded, its pinned copies exercised), untimed
    for k in range(max(3, args.warmup)):
        stage_inputs(k & 1, 0)
        stream.wait_event(copied[k & 1])
        step += 1
        F.wgrad_adamw_grouped(sets[k & 1], step=step, stream=stream, **HYPER)
        if layer.fp8_scales is not None:
            F.fp8_roll_scales(layer.fp8_scales, FP8_HEADROOM, stream=stream)
        consumed[k & 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    for ev in consumed:
        ev.record(stream)
    e0 = time.perf_counter()
    e_first = None
    stage_inputs(0, 0)
    for k in range(e2e_steps):
        step += 1
        b = k & 1
        stream.wait_event(copied[b])
        st_ev[k][0].record(stream)
        F.wgrad_adamw_grouped(sets[b], step=step, stream=stream, **HYPER)
        if layer.fp8_scales is not None:
            F.fp8_roll_scales(layer.fp8_scales, FP8_HEADROOM, stream=stream)
        st_ev[k][1].record(stream)
        consumed[b].record(stream)
        with torch.cuda.stream(stream):
            res_host[b].copy_(w_first[:2], non_blocking=True)
        res_ev[b].record(stream)
        if k + 1 < e2e_steps:         # issued while step k runs
            stage_inputs(1 - b, k + 1)
        if k >= 1:                    # step k-1's result, while step k runs
            res_ev[1 - b].synchronize()
            checked.append(bool(torch.isfinite(res_host[1 - b].float()).all()))
        if k == 0:
            res_ev[0].synchronize()
            checked.append(bool(torch.isfinite(res_host[0].float()).all()))
            e_first = time.perf_counter()
    res_ev[(e2e_steps - 1) & 1].synchronize()
    checked.append(bool(torch.isfinite(res_host[(e2e_steps - 1) & 1].float()).all()))
    st = F.device_error(stream)
    if st != 0 or not all(checked):
        raise RuntimeError(f"e2e: {F.status_string(st)}, finite results {all(checked)}")
    e1 = time.perf_counter()
    torch.cuda.synchronize()
    e2e_ms = (e1 - e0) * 1e3 / e2e_steps
    copy_ms = [a.elapsed_time(b) for a, b in cp_ev[1:]]
    comp_ms = [a.elapsed_time(b) for a, b in st_ev]
    # copies of step k+1 that ended before step k's compute did: hidden
    hidden = sum(1 for k in range(e2e_steps - 1)
                 if st_ev[k][1].elapsed_time(cp_ev[k + 1][1]) <= 0.0)
    e2e = dict(steps=e2e_steps,
               first_step_ms=(e_first - e0) * 1e3,
               later_steps_ms=(e1 - e_first) * 1e3 / max(1, e2e_steps - 1),
               h2d_gbs=layer.h2d_bytes() / (statistics.median(h2d_ms) * 1e-3) / 1e9,
               copy_ms_median=statistics.median(copy_ms) if copy_ms else None,
               compute_ms_median=statistics.median(comp_ms),
               copies_hidden_frac=hidden / max(1, e2e_steps - 1))
    if dist:
        e2e_ms, unf_ms = max_over_ranks([e2e_ms, unf_ms], dev)

    return dict(layer=layer, elapsed_ms=elapsed_ms, kern_ms=kern_ms, launch_ms=launch_ms,
                steady=steady, sampler=sampler, unf_ms=unf_ms,
                per_proj_ms=per_proj_ms, backward=backward, opt_ms=opt_ms, opt_fmt=sfmt,
                acc_ms=acc_ms, sr_ms=sr_ms,
                e2e=e2e, e2e_ms=e2e_ms, clocks=sampler.summary(w0, w1) if sampler else None,
                config=F.describe_config(bt, 4096, 4096, fmt))


def unfused_step(F, layer, step, dw):
    for it in layer.items:
        g = dw[:it["d_in"] * it["d_out"]].view(it["d_out"], it["d_in"])
        F.wgrad(it["x"], it["dy"], g)
        F.adamw(g, it["w"], it["m"], it["v"], step=step, m_scale=it["ms"], v_scale=it["vs"],
                **HYPER)


# ---------------------------------------------------------------------------
# the full linear stack (32 layers x 7 projections)
# ---------------------------------------------------------------------------

STACK_LAYERS = 32


class Stack:
    """All 224 projections of Llama-3.1-8B, generated on the device (seeded
    normal values of the same recipe; activations of this size are not drawn
    on the host).  As in the model, q, k, v read one X per layer and gate, up
    read one X per layer; o and down have their own."""

    def __init__(self, bt, fmt, dy_std, dev, seed=5000):
        from weight_gradient_gemm_gb300 import forge as F
        g = torch.Generator(device=dev)
        g.manual_seed(seed)

        def normal(shape, std):
            return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std
                    ).to(torch.bfloat16)

        self.bt, self.fmt = bt, fmt
        self.layers = []
        for _ in range(STACK_LAYERS):
            xs = {"attn": normal((bt, 4096), 1.0), "o": normal((bt, 4096), 1.0),
                  "mlp": normal((bt, 4096), 1.0), "down": normal((bt, 14336), 1.0)}
            which = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "mlp",
                     "up": "mlp", "down": "down"}
            items = []
            for name, d_out, d_in in LLAMA31_8B_SHAPES:
                m, v, ms, vs = F.alloc_moments(d_out, d_in, fmt, dev)
                items.append(dict(name=name, d_in=d_in, d_out=d_out, X=xs[which[name]],
                                  dY=normal((bt, d_out), dy_std), W=normal((d_out, d_in), 0.02),
                                  m=m, v=v, m_scale=ms, v_scale=vs))
            self.layers.append(items)

    def linears(self):
        return [it for layer in self.layers for it in layer]

    def flops(self):
        return sum(2.0 * self.bt * it["d_in"] * it["d_out"] for it in self.linears())

    def params(self):
        return sum(it["d_in"] * it["d_out"] for it in self.linears())

    def alg_bytes(self):
        # state once per linear; each distinct X once; each dY once
        state = sum(it["d_in"] * it["d_out"] * STATE_BYTES[self.fmt] for it in self.linears())
        xs = {id(it["X"]): it["X"].numel() * 2 for it in self.linears()}
        dys = sum(it["dY"].numel() * 2 for it in self.linears())
        return state + sum(xs.values()) + dys


def stack_step(F, stack, step, events=None, stream=None):
    """One optimizer step over the whole stack in backward order (layer 31
    first); each layer's seven projections are one grouped launch."""
    for i, layer in enumerate(reversed(stack.layers)):
        if events is not None:
            events[i][0].record(stream)
        F.wgrad_adamw_grouped(layer, step=step, **HYPER)
        if events is not None:
            events[i][1].record(stream)


def stack_unfused_step(F, stack, step, dw):
    for layer in reversed(stack.layers):
        for it in reversed(layer):        # down, up, gate, o, v, k, q
            g = dw[:it["d_in"] * it["d_out"]].view(it["d_out"], it["d_in"])
            F.wgrad(it["X"], it["dY"], g)
            F.adamw(g, it["W"], it["m"], it["v"], step=step, m_scale=it["m_scale"],
                    v_scale=it["v_scale"], **HYPER)


def run_stack(args, dev):
    """The full-stack workload: fused step vs the library's unfused path."""
    from weight_gradient_gemm_gb300 import forge as F
    F.lib()
    parts = args.workload.split("_")
    bt = int(parts[3][2:])
    fmt = {"fp32": 0, "bf16": 1, "int8": 2}[parts[4]]
    stack = Stack(bt, fmt, 1e-3, dev)
    stream = torch.cuda.current_stream()
    step = 0
    for _ in range(args.warmup):
        step += 1
        stack_step(F, stack, step)
    assert F.device_error() == 0
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(STACK_LAYERS)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index)
    time.sleep(0.25)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    t0.record(stream)
    for k in range(args.steps):
        step += 1
        stack_step(F, stack, step, ev[k], stream)
    t1.record(stream)
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    sampler.stop()
    st = F.device_error()
    if st != 0:
        raise RuntimeError(F.status_string(st))
    ms = t0.elapsed_time(t1) / args.steps
    kern_ms = sum(a.elapsed_time(b) for row in ev for (a, b) in row) / args.steps
    # the unfused path: forge_wgrad (bf16 dW) + forge_adamw per linear
    dw = torch.empty(max(it["d_in"] * it["d_out"] for it in stack.linears()),
                     dtype=torch.bfloat16, device=dev)
    step += 1
    stack_unfused_step(F, stack, step, dw)
    torch.cuda.synchronize()
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    unf_steps = max(2, min(args.steps, 5))
    u0.record(stream)
    for _ in range(unf_steps):
        step += 1
        stack_unfused_step(F, stack, step, dw)
    u1.record(stream)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    unf_ms = u0.elapsed_time(u1) / unf_steps

    peaks, peak_kind = measured_peaks()
    flops, byts = stack.flops(), stack.alg_bytes()
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    kern_s_per_launch = kern_ms * 1e-3 / STACK_LAYERS
    roof = roofline_of(flops / STACK_LAYERS, byts / STACK_LAYERS, kern_s_per_launch, peaks,
                       peak_kind)
    line = {
        "metric": METRIC, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded normal, generated on the device)",
        "config": {"workload": args.workload, "bt": bt, "moments": FMT_NAMES[fmt],
                   "linears": 7 * STACK_LAYERS, "params_per_step": stack.params(),
                   "order": "backward: layer 31 to 0, one grouped launch per layer",
                   "l2": f"inputs larger than L2: {byts / 1e9:.1f} GB per step"},
        "roofline": roof,
        "roofline_step": {"roofline_ms": max(t_hbm, t_tc) * 1e3,
                          "frac_of_roofline": max(t_hbm, t_tc) * 1e3 / ms},
        "unfused": {"ms_per_step": unf_ms, "fused_speedup": unf_ms / ms,
                    "path": "forge_wgrad (bf16 dW) + forge_adamw, 448 launches per step"},
        "gpu_launches": STACK_LAYERS * args.steps,
        "clocks": sampler.summary(w0, w1),
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# the other configurations of the metric, each timed in the same run
# ---------------------------------------------------------------------------

def _device_normal(g, shape, std, dev):
    return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std
            ).to(torch.bfloat16)


def device_layer(bt, fmt, dy_std, spike, dev, seed):
    """One layer's seven projections with inputs drawn on the device (the
    recipe's distributions: X ~ N(0,1), dY ~ N(0, dy_std) with floor(spike*BT)
    token rows x100, W ~ N(0, 0.02)); each projection has its own X."""
    from weight_gradient_gemm_gb300 import forge as F
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    group = []
    scales = F.alloc_fp8_scales(14, device=dev) if fmt == 3 else None
    for i, (name, d_out, d_in) in enumerate(LLAMA31_8B_SHAPES):
        dy = torch.randn((bt, d_out), generator=g, device=dev, dtype=torch.float32) * dy_std
        n = int(math.floor(spike * bt))
        if n:
            dy[torch.randperm(bt, generator=g, device=dev)[:n]] *= 100.0
        m, v, ms, vs = F.alloc_moments(d_out, d_in, fmt, dev)
        if scales is not None:
            ms, vs = scales[2 * i], scales[2 * i + 1]
        group.append(dict(X=_device_normal(g, (bt, d_in), 1.0, dev), dY=dy.to(torch.bfloat16),
                          W=_device_normal(g, (d_out, d_in), 0.02, dev), m=m, v=v,
                          m_scale=ms, v_scale=vs))
    return group, scales


def roofline_of(flops, nbytes, launch_s, peaks, peak_kind, traffic=None):
    """The roofline object of one launch: bound by whichever of the tensor
    time (burst cuBLAS bf16 peak: every timed region here is tens of
    milliseconds, a burst) or the HBM time (measured copy bandwidth) is
    larger; `frac_sustained` gives the tensor fraction against the sustained
    figure as well."""
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        ach = nbytes / launch_s / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "traffic": traffic,
                "peak_kind": f"{peak_kind} (copy bandwidth)"}
    ach = flops / launch_s / 1e12
    sus = peaks.get("bf16_tflops_sustained")
    return {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": ach / peaks["bf16_tflops"], "traffic": traffic,
            "peak_kind": f"{peak_kind} (cuBLAS bf16, burst)",
            "frac_sustained": ach / sus if sus else None}


def launch_stats(ms):
    return {"launches": len(ms), "median_ms": statistics.median(ms), "min_ms": min(ms),
            "max_ms": max(ms), "mean_ms": sum(ms) / len(ms)}


def timed_launches(fn, n, stream):
    """n calls of fn, each bracketed by CUDA events on `stream`; returns the
    per-launch milliseconds and the wall-clock window."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    return [a.elapsed_time(b) for a, b in ev], w0, w1


# (block name, workload it measures, BT, moment format, spike fraction)
TENSOR_BLOCKS = [
    ("c3_bt512_bf16", "llama31_8b_layer_bt512_bf16", 512, 1, 0.01),
    ("int8_bt512", "llama31_8b_layer_bt512_int8", 512, 2, 0.0),
    ("fp8_bt512", "llama31_8b_layer_bt512_fp8", 512, 3, 0.0),
    ("c3_bt2048_bf16", "llama31_8b_layer_bt2048_bf16", 2048, 1, 0.01),
    ("c4_bt4096_int8", "llama31_8b_layer_bt4096_int8", 4096, 2, 0.0),
    ("bt4096_fp32", "llama31_8b_layer_bt4096_fp32", 4096, 0, 0.0),
    ("c3_bt8192_bf16", "llama31_8b_layer_bt8192_bf16", 8192, 1, 0.01),
]


def dgrad_block(F, group, bt, n, stream, sampler, peaks):
    """dX = dY W for the seven projections at a tensor-bound token count: one
    forge_dgrad_grouped launch (caller workspace) against cuBLAS's seven
    torch.matmul calls on the same tensors, each timed per step with CUDA
    events, alternating three rounds so both see the same clocks."""
    dx = [torch.empty((bt, g["W"].shape[1]), dtype=torch.bfloat16, device=g["W"].device)
          for g in group]
    items = [dict(dY=g["dY"], W=g["W"], dX=o) for g, o in zip(group, dx)]
    ws_bytes = F.dgrad_workspace_bytes(items)
    ws = (torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=dx[0].device)
          if ws_bytes else None)

    def forge_dx():
        F.dgrad_grouped(items, workspace=ws)

    def cublas_dx():
        for g, o in zip(group, dx):
            torch.matmul(g["dY"], g["W"], out=o)
    for _ in range(3):
        forge_dx()
        cublas_dx()
    f_ms, c_ms, f_win = [], [], []
    for _ in range(3):
        ms, w0, w1 = timed_launches(forge_dx, max(10, n // 3), stream)
        f_ms += ms
        f_win.append((w0, w1))
        ms, _, _ = timed_launches(cublas_dx, max(10, n // 3), stream)
        c_ms += ms
    if F.device_error() != 0:
        raise RuntimeError("dgrad block: device error")
    flops = sum(2.0 * bt * g["W"].numel() for g in group)
    f_med, c_med = statistics.median(f_ms), statistics.median(c_ms)
    tf = flops / (f_med * 1e-3) / 1e12
    del dx, items, ws
    return {"launch": "forge_dgrad_grouped: the seven projections in one launch",
            "ms_per_step": f_med, "tflops": tf,
            "frac": tf / peaks["bf16_tflops"], "per_launch": launch_stats(f_ms),
            "workspace_bytes": ws_bytes,
            "cublas_ms_per_step": c_med, "vs_cublas": c_med / f_med,
            "clocks": sampler.summary(f_win[0][0], f_win[-1][1])}


def config_blocks(args, dev, peaks, peak_kind):
    """The metric's other Llama-3.1-8B configurations, each timed in-process
    with CUDA events around every grouped launch (at least ~0.3 s of
    launches, so the clock sampler sees them), with its own roofline, clocks
    and stored ncu traffic: fp8 moments at 512 tokens (HBM-bound; each step
    is the grouped launch plus the scale roll), C3 at 2048 and 8192 tokens
    (bf16 moments), C4 at 4096 (int8), fp32 moments at 4096, and C5 (the
    224-linear stack at 512 and 8192 tokens, fp32 moments, one grouped launch
    per layer).  The 4096-token fp32 block also times the layer's input
    gradient (dgrad_block)."""
    from weight_gradient_gemm_gb300 import forge as F
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(dev.index)
    time.sleep(0.25)
    out = {}
    for name, workload, bt, fmt, spike in TENSOR_BLOCKS:
        group, f8 = device_layer(bt, fmt, 1e-3, spike, dev, seed=7000 + bt + fmt)
        step = [0]

        def one():
            step[0] += 1
            F.wgrad_adamw_grouped(group, step=step[0], **HYPER)
            if f8 is not None:
                F.fp8_roll_scales(f8, FP8_HEADROOM)
        for _ in range(max(args.warmup, 3) + 10):   # moments warmed by 10 prior steps
            one()
        warm_ms, _, _ = timed_launches(one, 3, stream)
        n = max(args.steps, math.ceil(300.0 / max(statistics.median(warm_ms), 1e-3)))
        ms, w0, w1 = timed_launches(one, n, stream)
        if F.device_error() != 0:
            raise RuntimeError(f"{name}: device error")
        flops = sum(2.0 * bt * g["W"].numel() for g in group)
        nbytes = sum(g["W"].numel() * STATE_BYTES[fmt]
                     + 2.0 * bt * (g["X"].shape[1] + g["dY"].shape[1]) for g in group)
        mean_s = sum(ms) / len(ms) * 1e-3
        # cuBLAS's plain weight-gradient GEMM dW = dY^T X (bf16 out) on the
        # same tensors, timed the same way right after: the main loop's
        # reference under the same clocks and power
        cub = None
        if bt >= 2048:
            outs = [torch.empty_like(g["W"]) for g in group]

            def cublas_wgrad():
                for g, o in zip(group, outs):
                    torch.matmul(g["dY"].t(), g["X"], out=o)
            for _ in range(3):
                cublas_wgrad()
            cms, c0, c1 = timed_launches(cublas_wgrad, max(10, n // 2), stream)
            cmean = sum(cms) / len(cms) * 1e-3
            cub = {"ms_per_step": cmean * 1e3, "tflops": flops / cmean / 1e12,
                   "fused_vs_cublas_gemm": cmean / mean_s, "clocks": sampler.summary(c0, c1)}
            del outs
        dgrad = dgrad_block(F, group, bt, n, stream, sampler, peaks) if bt == 4096 and fmt == 0 \
            else None
        out[name] = {"workload": workload, "bt": bt, "moments": FMT_NAMES[fmt],
                     "launch": "forge_wgrad_adamw_grouped, seven projections",
                     "kernel": F.describe_config(bt, 4096, 4096, fmt),
                     "tflops": flops / mean_s / 1e12,
                     "roofline": roofline_of(flops, nbytes, mean_s, peaks, peak_kind,
                                             stored_traffic(workload)),
                     "per_launch": launch_stats(ms), "clocks": sampler.summary(w0, w1),
                     "cublas_wgrad_gemm": cub}
        if dgrad is not None:
            out[name]["dgrad"] = dgrad
        del group, f8
        torch.cuda.empty_cache()
    # C5: the whole stack at 512 and 8192 tokens
    for sbt in (512, 8192):
        stack = Stack(sbt, 0, 1e-3, dev)
        step = [0]

        def stack_once():
            step[0] += 1
            stack_step(F, stack, step[0])
        for _ in range(max(args.warmup, 3)):
            stack_once()
        n = max(3, min(args.steps, 10))
        ms, w0, w1 = timed_launches(stack_once, n, stream)
        if F.device_error() != 0:
            raise RuntimeError("stack: device error")
        flops, nbytes = stack.flops(), stack.alg_bytes()
        mean_s = sum(ms) / len(ms) * 1e-3
        out[f"c5_stack_bt{sbt}_fp32"] = {
            "workload": f"llama31_8b_stack_bt{sbt}_fp32", "bt": sbt, "moments": "fp32",
            "launch": "32 forge_wgrad_adamw_grouped launches per step, backward order",
            "ms_per_step": mean_s * 1e3, "tflops": flops / mean_s / 1e12,
            "roofline": roofline_of(flops / STACK_LAYERS, nbytes / STACK_LAYERS,
                                    mean_s / STACK_LAYERS, peaks, peak_kind),
            "per_step": launch_stats(ms), "clocks": sampler.summary(w0, w1)}
        del stack
        torch.cuda.empty_cache()
    sampler.stop()
    return out


# ---------------------------------------------------------------------------
# the CPU oracle (reported baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(workload: str, rows: int):
    """Inputs for one oracle step on the first `rows` weight rows of each of
    the seven projections."""
    import oracle as O
    cfg, bt, fmt, dy_std, spike = workload_spec(workload)
    out = []
    for i, (name, d_out, d_in) in enumerate(LLAMA31_8B_SHAPES):
        s = make_step_inputs(cfg, i, 0, bt, d_in, d_out, dy_std=dy_std, with_w=True,
                             spike_frac=spike)
        r = min(rows, d_out)
        out.append(dict(x=bf16_bits(s.x), dy=bf16_bits(s.dy)[:, :r].copy(),
                        w=bf16_bits(s.w)[:r].copy(), m=O.zero_moment(fmt, r, d_in),
                        v=O.zero_moment(fmt, r, d_in), r=r, d_in=d_in))
    return out, bt


def oracle_step(sample, t):
    import oracle as O
    h = O.Hyper(lr=HYPER["lr"], beta1=HYPER["beta1"], beta2=HYPER["beta2"], eps=HYPER["eps"],
                wd=HYPER["weight_decay"])
    for s in sample:
        O.step(s["x"], s["dy"], s["w"], s["m"], s["v"], h, t)


def oracle_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def _oracle_rows_for(workload: str, target_s: float) -> int:
    """Rows per projection for an oracle step of about target_s seconds: a
    two-point fit (fixed cost of decoding X plus a cost per weight row)."""
    times = {}
    for r in (16, 64):
        sample, _ = oracle_sample(workload, r)
        t0 = time.perf_counter()
        oracle_step(sample, 1)
        times[r] = time.perf_counter() - t0
    per_row = max((times[64] - times[16]) / 48.0, 1e-7)
    fixed = max(times[16] - 16 * per_row, 0.0)
    return max(1, min(14336, int((target_s - fixed) / per_row)))


def time_oracle(workload: str, target_s: float):
    """Oracle TFLOP/s on a row sample sized for about target_s seconds."""
    rows = _oracle_rows_for(workload, target_s)
    sample, bt = oracle_sample(workload, rows)
    t0 = time.perf_counter()
    oracle_step(sample, 1)
    dt = time.perf_counter() - t0
    flops = sum(2.0 * bt * s["r"] * s["d_in"] for s in sample)
    return flops / dt / 1e12, dt, rows, bt


def run_metadata():
    """What the line was measured on: GPU name, driver and CUDA versions,
    PyTorch version, the kernel sources' hash and the host's core count.
    Never raises: a field that cannot be read is null."""
    out = {"gpu": None, "driver": None, "cuda": None, "torch": torch.__version__,
           "kernel_sources": None, "host_cores": os.cpu_count()}
    try:
        out["kernel_sources"] = source_digest()
    except Exception:
        pass
    try:
        out["cuda"] = torch.version.cuda
        if torch.cuda.is_available():
            out["gpu"] = torch.cuda.get_device_name(torch.cuda.current_device())
    except Exception:
        pass
    try:
        r = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=10)
        if r.returncode == 0 and r.stdout.strip():
            out["driver"] = r.stdout.strip().splitlines()[0]
    except Exception:
        pass
    return out


def cpu_baseline_block(workload):
    # the two-point fit overestimates the cost per row of larger samples: a
    # 20 s target lands at about 10-12 s of oracle work
    value, dt, rows, bt = time_oracle(workload, 20.0)
    return {"value": value, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": (f"one fp64 oracle step (numpy: BLAS matmul for G, then AdamW and rounding)"
                       f" on the first {rows} rows of each of the 7 projections at BT={bt}, "
                       f"{dt:.1f} s")}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample
    of the same workload each step."""
    cfg, bt, fmt, dy_std, spike = workload_spec(args.workload)
    budget_s = args.reference_budget
    per_step = budget_s / max(1, args.steps + args.warmup)
    rows = _oracle_rows_for(args.workload, 0.6 * per_step)   # the fit runs slightly short
    sample, bt = oracle_sample(args.workload, rows)
    for t in range(args.warmup):
        oracle_step(sample, t + 1)
    t0 = time.perf_counter()
    for t in range(args.steps):
        oracle_step(sample, args.warmup + t + 1)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    flops = sum(2.0 * bt * s["r"] * s["d_in"] for s in sample)
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "bt": bt, "moments": FMT_NAMES[fmt],
                   "sample_rows_per_projection": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle_threads(),
                         "kind": "oracle",
                         "sample": f"first {rows} rows of each of the 7 projections per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------

def optimizers_block(opt_ms, sfmt, layer, peaks):
    """The other fused optimizers (diagnostic): one forge_wgrad_opt launch per
    projection, the step's time and its HBM roofline fraction; bytes per
    parameter = W read + write (4) + 2 x state element size per state."""
    names = ["sgd", "sgd_momentum", "adagrad", "rmsprop", "lion", "nadam", "radam"]
    eb = 4 if sfmt == 0 else 2
    operands = layer.h2d_bytes()
    out = {"states": "fp32" if sfmt == 0 else "bf16",
           "launch": "forge_wgrad_opt_grouped, one launch per layer", "peak_gbs": peaks["hbm_gbs"]}
    for opt, name in enumerate(names):
        nst = [0, 1, 1, 1, 1, 2, 2][opt]
        ms = opt_ms[opt]
        nbytes = layer.params() * (4 + 2 * eb * nst) + operands
        out[name] = {"ms_per_step": ms, "gbs": nbytes / (ms * 1e-3) / 1e9,
                     "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    return out


def accumulate_block(acc_ms, layer, peaks):
    """The accumulate mode (diagnostic): B = beta B + dY^T X into fp32 for the
    seven projections, one launch each; bytes per parameter 8 with beta = 1
    (B read and written), 4 with beta = 0, plus the operands."""
    out = {"launch": "forge_wgrad_accumulate_grouped, one launch per layer",
           "peak_gbs": peaks["hbm_gbs"]}
    for beta, per in ((1.0, 8), (0.0, 4)):
        ms = acc_ms[beta]
        nbytes = layer.params() * per + layer.h2d_bytes()
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[f"beta_{int(beta)}"] = {"ms_per_step": ms, "gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]}
    if "final" in acc_ms:
        # the final micro-batch's step: the state stream plus B read (4 bytes)
        ms = acc_ms["final"]
        nbytes = layer.params() * (STATE_BYTES[layer.fmt] + 4) + layer.h2d_bytes()
        gbs = nbytes / (ms * 1e-3) / 1e9
        out["final_step"] = {
            "launch": "forge_wgrad_adamw_acc_grouped: AdamW on fp32(B + dY^T X), one launch",
            "ms_per_step": ms, "gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
            "accumulate_then_adamw_ms": acc_ms["final_unfused"],
            "speedup": acc_ms["final_unfused"] / ms}
    return out


def backward_block(bw, flops, fused_ms, peaks, peak_kind):
    """The backward-step diagnostic: dX = dY W for the seven projections
    (the same FLOPs as the weight gradient) in one forge_dgrad_grouped launch
    against the bf16 tensor peak (burst), next to one forge_dgrad per
    projection and cuBLAS on the same tensors, and the whole step as
    forge_linear_backward_grouped (one grouped dX launch, then one grouped
    fused launch)."""
    peak = peaks["bf16_tflops"]
    dgrad_tf = flops / (bw["dgrad_ms"] * 1e-3) / 1e12
    return {
        "dgrad": {"ms_per_step": bw["dgrad_ms"], "tflops": dgrad_tf,
                  "roofline": {"bound": "tensor", "achieved": dgrad_tf, "peak": peak,
                               "unit": "TFLOP/s", "frac": dgrad_tf / peak,
                               "peak_kind": f"{peak_kind} (cuBLAS bf16, burst)"},
                  "launch": "forge_dgrad_grouped: the seven projections in one launch",
                  "per_projection_ms_per_step": bw.get("dgrad_each_ms"),
                  "workspace_bytes": bw.get("workspace_bytes"),
                  "kernel_gate_up": bw["dgrad_config"],
                  "cublas_ms_per_step": bw["cublas_dgrad_ms"],
                  "vs_cublas": bw["cublas_dgrad_ms"] / bw["dgrad_ms"]},
        "ms_per_step": bw["linear_backward_ms"],
        "tflops": 2.0 * flops / (bw["linear_backward_ms"] * 1e-3) / 1e12,
        "fused_step_ms": fused_ms,
        "vs_fused_step": bw["linear_backward_ms"] / fused_ms,
        "path": "forge_linear_backward_grouped: one grouped dX launch, then one grouped "
                "fused launch",
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="forge", choices=["forge", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="one of %s, llama31_8b_layer_bt<BT>_<fp32|bf16|int8>, or the full "
                         "224-linear stack llama31_8b_stack_bt<BT>_<fp32|bf16|int8>" % sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-diagnostics", action="store_true",
                    help="time the step only (no steady repeat, unfused arm, backward, other "
                         "optimizers, accumulate, SR store or e2e): for profiling runs")
    ap.add_argument("--no-blocks", action="store_true",
                    help="skip the other configurations (C3, C4, fp32 at 4096, the C5 stack)")
    ap.add_argument("--reference-budget", type=float, default=120.0,
                    help="seconds of oracle work the reference arm aims for (all steps)")
    ap.add_argument("--only", default="",
                    help="comma-separated projections (q,k,v,o,gate,up,down) for small profiling "
                         "runs; the JSON line then describes that subset")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    if args.workload.startswith("llama31_8b_stack_"):
        if world > 1:
            raise SystemExit("the stack workload runs on one GPU")
        run_stack(args, dev)
        return
    res = run_gpu(args, rank, world, dev)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return

    layer = res["layer"]
    cfg, bt, fmt, dy_std, spike = workload_spec(args.workload)
    peaks, peak_kind = measured_peaks()
    ms = res["elapsed_ms"] / args.steps
    flops = layer.flops()
    value = job_value(world, flops, ms * 1e-3) / 1e12
    launches = args.steps * (2 if fmt == 3 else 1)   # the grouped launch (+ fp8 scale roll)
    kern_s_per_launch = res["kern_ms"] * 1e-3 / args.steps
    t_hbm = layer.alg_bytes() / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    roof = roofline_of(flops, layer.alg_bytes(), kern_s_per_launch, peaks, peak_kind,
                       stored_traffic(args.workload))
    roofline_time = max(t_hbm, t_tc)
    steady = None
    if res["steady"] is not None:
        sd = res["steady"]
        lm = sd["launch_ms"]
        q = len(lm) // 4
        span = sd["w1"] - sd["w0"]
        quarters = []
        for i in range(4):
            part = lm[i * q:(i + 1) * q] if i < 3 else lm[3 * q:]
            cs = res["sampler"].summary(sd["w0"] + i * span / 4, sd["w0"] + (i + 1) * span / 4)
            quarters.append({"median_ms": statistics.median(part), "sm_mhz": cs["sm_mhz"],
                             "samples": cs.get("samples")})
        runs = [statistics.median(lm[i * 20:(i + 1) * 20]) for i in range(3) if len(lm) >= 20 * (i + 1)]
        steady = {"what": "the same grouped launch repeated for about 1 s after the timed region",
                  **launch_stats(lm),
                  "protocol_3x20_medians_ms": runs,
                  "protocol_note": "3 runs x median of 20 launches after at least 35 earlier "
                                   "launches (10 moment warm-up, the warm-up and the timed steps)",
                  "roofline_frac_median": roofline_of(flops, layer.alg_bytes(),
                                                      statistics.median(lm) * 1e-3, peaks,
                                                      peak_kind)["frac"],
                  "clocks": res["sampler"].summary(sd["w0"], sd["w1"]),
                  "by_quarter": quarters}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "bt": bt, "moments": FMT_NAMES[fmt],
                   "projections": [it["name"] for it in layer.items],
                   "params_per_step": layer.params(),
                   "l2": f"inputs larger than L2: {layer.alg_bytes() / 1e9:.2f} GB streamed per "
                         f"step vs {L2_BYTES / 2 ** 20:.0f} MiB L2",
                   "parallelism": "replicas" if world > 1 else "single",
                   "launch": "forge_wgrad_adamw_grouped: the seven projections in one launch",
                   "kernel": res["config"]},
        "roofline": roof,
        "roofline_step": {"roofline_ms": roofline_time * 1e3,
                          "frac_of_roofline": roofline_time * 1e3 / ms,
                          "params_per_s": layer.params() / (ms * 1e-3) * world,
                          "hbm_gbs": layer.alg_bytes() / (ms * 1e-3) / 1e9},
        "per_launch": launch_stats(res["launch_ms"]),
        "steady": steady,
        "gpu_launches": launches,
        "clocks": res["clocks"],
        "system": run_metadata(),
    }
    if not args.no_diagnostics:
        line.update({
            "unfused": {"ms_per_step": res["unf_ms"],
                        "value": job_value(world, flops, res["unf_ms"] * 1e-3) / 1e12,
                        "fused_speedup": res["unf_ms"] / ms,
                        "path": "forge_wgrad (bf16 dW) + forge_adamw"},
            "e2e": {"value": job_value(world, flops, res["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": res["e2e_ms"], "h2d_bytes_per_step": layer.h2d_bytes(),
                    "d2h_bytes_per_step": 4,
                    "pipeline": "X, dY of step k+1 copied from pinned host memory on a second "
                                "stream while step k computes; 4 bytes of each step's new W copied "
                                "to pinned memory and read by the host one step later (while "
                                "the next step runs); the library's status word checked at the "
                                "end; untimed warm-up steps first",
                    **res["e2e"]},
            "per_projection_separate_launches": [
                {"name": it["name"], "shape": [it["d_out"], it["d_in"]],
                 "us": round(t * 1e3, 2),
                 "gbs": round((it["d_in"] * it["d_out"] * STATE_BYTES[fmt]
                               + 2.0 * bt * (it["d_in"] + it["d_out"])) / (t * 1e-3) / 1e9, 1),
                 "tflops": round(2.0 * bt * it["d_in"] * it["d_out"] / (t * 1e-3) / 1e12, 1)}
                for it, t in zip(layer.items, res["per_proj_ms"])],
            "linear_backward": backward_block(res["backward"], flops, ms, peaks, peak_kind),
            "optimizers": optimizers_block(res["opt_ms"], res["opt_fmt"], layer, peaks),
            "accumulate": accumulate_block(res["acc_ms"], layer, peaks),
            "sr_store": None if res["sr_ms"] is None else {
                "ms_per_step": res["sr_ms"],
                "round_to_nearest_ms_per_step": sum(res["per_proj_ms"]),
                "overhead": res["sr_ms"] / sum(res["per_proj_ms"]) - 1.0,
                "launch": "forge_wgrad_adamw_sr_grouped (one launch per layer), against "
                          "forge_wgrad_adamw per projection",
                "vs_grouped_round_to_nearest": res["sr_ms"] / ms},
        })
    if not args.no_blocks and world == 1:
        del layer, res
        torch.cuda.empty_cache()
        line["configs"] = config_blocks(args, dev, peaks, peak_kind)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline_block(args.workload)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
