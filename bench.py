#!/usr/bin/env python3
"""Benchmark of the trellis-coded linear layers on GB300.

Workload (one step): the axis-1 decode-fused matvec at the MLP up-projection
shape R=17408 out rows x C=5120 in cols, L=16, T=256, for every k in {2,3,4}
and every M in {1,2,3,4} -- twelve launches over packed weights.  `value` is
the packed-weight bytes of those twelve launches divided by the step time
(GB/s); the prefill GEMM (R=17408, C=5120, k=2, M=2048) is timed in the same
run and reported as TFLOP/s under "prefill".

Inputs are seeded and synthetic (uniform random code words, fp16 scales
U[0.005, 0.02], bf16 x ~ N(0,1)).  Code buffers rotate through a set larger
than twice the L2 cache, so every launch streams its weights from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--extra]

Under torchrun every rank runs the same per-GPU workload (weak scaling); the
reported time is the maximum over ranks and `value` sums all ranks' bytes.
`--impl reference` times the oracle (plain C, one host core) on a bounded
sample of rows of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed-weight HBM GB/s (frac of GB300 peak) at M=1..4; prefill TFLOP/s at M=2048"
R, C, L, T = 17408, 5120, 16, 256
KS, MS = (2, 3, 4), (1, 2, 3, 4)
PREFILL_M = 2048
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def packed_bytes(k: int) -> int:
    return R * C * k // 8


def workload_desc():
    return {"workload": "axis-1 trellis matvec (MLP up-projection shape)", "rows": R, "cols": C, "k": list(KS),
            "L": L, "T": T, "M": list(MS), "launches_per_step": len(KS) * len(MS),
            "l2": "code buffers rotate through a set larger than 2x L2 (inputs exceed L2)"}


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _dev_words(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev)


def _dev_f16(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).to(dev)


def _dev_bf16(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def run_gpu(args):
    import torch
    import torch.distributed as tdist

    from trellis_coded_weight_gb300 import binding as tb
    from trellis_coded_weight_gb300 import build as tbuild
    from trellis_coded_weight_gb300 import inputs

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(tbuild.LIB):
        tbuild.build()
    if world > 1:
        tdist.barrier()
    tb.load()
    stream = torch.cuda.current_stream(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 132 << 20))

    # ---- inputs: rotating code sets (larger than 2x L2 per k), scales, x ----
    bufs, scales, geoms = {}, {}, {}
    for k in KS:
        nrot = int(2 * l2 // packed_bytes(k)) + 2
        bufs[k] = [_dev_words(inputs.random_words(inputs.SEED_CODES + 100 * k + i + 7919 * rank, (R, C * k // 32)), dev)
                   for i in range(nrot)]
        scales[k] = _dev_f16(inputs.uniform_f16(inputs.SEED_SCALES + k, (R,)), dev)
        geoms[k] = tb.Geometry(k, L, T, 1, R, C)
    xs = {M: _dev_bf16(inputs.normal_bf16(inputs.SEED_X + M, (M, C)), dev) for M in MS}
    outs = {M: torch.empty((M, R), dtype=torch.bfloat16, device=dev) for M in MS}
    rot = {k: 0 for k in KS}

    def launch(k, M):
        i = rot[k]
        rot[k] = (i + 1) % len(bufs[k])
        tb.matvec_axis1(bufs[k][i], scales[k], xs[M], geoms[k], outs[M])

    def step(events=None):
        for k in KS:
            for M in MS:
                if events is not None:
                    events[(k, M)][0].record(stream)
                launch(k, M)
                if events is not None:
                    events[(k, M)][1].record(stream)

    def sync_all():
        torch.cuda.synchronize(dev)
        if world > 1:
            tdist.barrier()

    for _ in range(args.warmup):
        step()
    # ---- timed region: exactly K steps, per-launch events on the launch stream ----
    ev = {(k, M): [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
          for k in KS for M in MS}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sync_all()
    with ClockSampler(local) as clk:
        t0.record(stream)
        for s in range(args.steps):
            step({key: ev[key][s] for key in ev})
        t1.record(stream)
        sync_all()
    ms_total = t0.elapsed_time(t1)
    if world > 1:
        tt = torch.tensor([ms_total], device=dev, dtype=torch.float64)
        tdist.all_reduce(tt, op=tdist.ReduceOp.MAX)
        ms_total = float(tt.item())
    per_launch = {key: statistics.median(e[0].elapsed_time(e[1]) for e in ev[key]) for key in ev}
    step_bytes = sum(packed_bytes(k) for k in KS for M in MS)
    value = world * step_bytes * args.steps / (ms_total * 1e-3) / 1e9

    # ---- end to end through the C ABI with host buffers (x in, out back) ----
    x_host = {M: xs[M].cpu().pin_memory() for M in MS}
    o_host = {M: torch.empty((M, R), dtype=torch.bfloat16).pin_memory() for M in MS}
    x_dev = {M: torch.empty_like(xs[M]) for M in MS}

    def e2e_step():
        for k in KS:
            for M in MS:
                x_dev[M].copy_(x_host[M], non_blocking=True)
                i = rot[k]
                rot[k] = (i + 1) % len(bufs[k])
                tb.matvec_axis1(bufs[k][i], scales[k], x_dev[M], geoms[k], outs[M])
                o_host[M].copy_(outs[M], non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    sync_all()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        e2e_step()
    b.record(stream)
    sync_all()
    e2e_ms = a.elapsed_time(b)
    if world > 1:
        tt = torch.tensor([e2e_ms], device=dev, dtype=torch.float64)
        tdist.all_reduce(tt, op=tdist.ReduceOp.MAX)
        e2e_ms = float(tt.item())
    h2d = sum(M * C * 2 for k in KS for M in MS)
    d2h = sum(M * R * 2 for k in KS for M in MS)
    e2e = {"value": world * step_bytes * args.steps / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    prefill = run_prefill(args, dev, stream, tb, inputs)
    res = dict(value=value, ms_total=ms_total, per_launch=per_launch, e2e=e2e, clocks=clk.summary(),
               prefill=prefill, world=world, rank=rank, launches=len(KS) * len(MS) * args.steps)
    if args.extra:
        res["extra"] = run_extra(args, dev, stream, tb, inputs, l2)
    if world > 1:
        tdist.barrier()
        tdist.destroy_process_group()
    return res
