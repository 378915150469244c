#!/usr/bin/env python3
"""Benchmark of the trellis-coded linear layers on GB300.

Headline (one step): the axis-1 decode-fused matvec at the MLP up-projection
shape R=17408 out rows x C=5120 in cols, L=16, T=256, for every k in {2,3,4}
and every M in {1,2,3,4} -- twelve launches over packed weights.  `value` is
the packed-weight bytes of those twelve launches divided by the step time
(GB/s), timed over exactly --steps steps.

The same run times every other row of the hot path at its full size, each in
`breakdown` with its median and p10/p90 launch time, its algorithmic bytes or
FLOPs and its fraction of the measured peak: the fused gate/up SwiGLU layer
(two 17408 x 5120 matrices, k = 2, 3), the axis-0 down projection (stored
W^T 17408 x 5120, k = 2, 3), the bf16 expansion (k = 2..4), the prefill GEMM
(k = 2, M = 8 / 16 / 24 / 32 / 512 / 2048, next to expand + cuBLAS), the axis-0
prefill (k = 3, M = 8 / 32 / 64 / 512 / 2048, next to expand + cuBLAS), the decode
MLP block as a CUDA graph, and two load-only floors of the packed stream.

`e2e` is the headline's twelve launches through trellis_matvec_axis1_host, one
C call per launch that brings its x in from pinned host memory and its output
back (through the buffers' device mapping), on one stream; `e2e.two_streams` the same calls alternating between two
streams.  `roofline` is the axis-1 matvec's: algorithmic bytes per launch over
the timed region's mean launch time, against the measured HBM copy rate.

Inputs are seeded and synthetic (uniform random code words, fp16 scales
U[0.005, 0.02], bf16 x ~ N(0,1), or N(0, 0.5) for the axis-0 input).  Code
buffers rotate through a set larger than twice the L2 cache, so every launch
streams its weights from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs the same per-GPU workload (weak scaling); the
reported time is the maximum over ranks and `value` sums all ranks' bytes.
`--impl reference` times the oracle (plain C, one host core) on a bounded
sample of rows of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
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
PREFILL_M = (8, 16, 24, 32, 512, 2048)  # up to 24: the register-decode path; 32 and up: tcgen05
PREFILL0_M = (8, 32, 64, 512, 2048)  # up to 32: the register-decode path; 64 and up: tcgen05
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
    """Samples nvidia-smi clocks and throttle reasons while running; every
    sample carries its host time, so a window (the timed region) can be
    summarised on its own."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index, self.proc, self.samples = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
            time.sleep(0.3)  # the first sample arrives before the measured work starts
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            reasons = {nm for nm, v in zip(self.NAMES, parts[3:7]) if v.lower() == "active"}
            self.samples.append((time.time(), sm, mx, reasons))

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, window=None):
        s = self.samples if window is None else [x for x in self.samples if window[0] <= x[0] <= window[1]]
        if not s:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(x[1] for x in s), "sm_max_mhz": max(x[2] for x in s),
                "reasons": sorted(set().union(*(x[3] for x in s))), "samples": len(s)}


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


class Timer:
    """Launch timing on the launching stream with CUDA events: a batch of n launches bracketed by two events
    (the mean), and per-launch event pairs (p10/p90).  A short device sleep ahead of each batch lets the host
    queue the launches, so no host gaps fall inside it."""

    def __init__(self, torch, dev, stream, n):
        self.torch, self.dev, self.stream, self.n = torch, dev, stream, n

    def __call__(self, fn, nrot=1):
        torch = self.torch
        for i in range(3):
            fn(i % nrot)
        torch.cuda.synchronize(self.dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(5e6))
        a.record(self.stream)
        for i in range(self.n):
            fn(i % nrot)
        b.record(self.stream)
        torch.cuda.synchronize(self.dev)
        mean_ms = a.elapsed_time(b) / self.n
        es = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(self.n)]
        torch.cuda._sleep(int(5e6))
        for i in range(self.n):
            es[i][0].record(self.stream)
            fn(i % nrot)
            es[i][1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        ts = sorted(x.elapsed_time(y) for x, y in es)
        return {"us": mean_ms * 1e3, "us_p10_p90": [ts[int(0.1 * (len(ts) - 1))] * 1e3, ts[int(0.9 * (len(ts) - 1))] * 1e3]}


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

    # ---- inputs of the headline: rotating code sets (larger than 2x L2 per k), scales, x ----
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
    # The headline calls the C entry point directly with its arguments prepared once (pointers, geometry,
    # stream), so that the host issues launches faster than the GPU runs them; the e2e leg below goes through
    # the Python binding.  The binding's own checks ran on these tensors during set-up.
    lib = tb.load()
    sptr = stream.cuda_stream
    cargs = {}
    for k in KS:
        for M in MS:
            tb.matvec_axis1(bufs[k][0], scales[k], xs[M], geoms[k], outs[M])
            for i, b in enumerate(bufs[k]):
                cargs[(k, M, i)] = (b.data_ptr(), scales[k].data_ptr(), xs[M].data_ptr(), outs[M].data_ptr(), M,
                                    ctypes.byref(geoms[k].c()), sptr)
    fn_mv = lib.trellis_matvec_axis1

    def launch(k, M):
        i = rot[k]
        rot[k] = (i + 1) % len(bufs[k])
        st = fn_mv(*cargs[(k, M, i)])
        if st:
            raise RuntimeError(f"trellis_matvec_axis1 returned {st}")

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

    res = {"world": world, "rank": rank}
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            step()
        # ---- timed region: exactly K steps, one event pair around them ----
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sync_all()
        h0 = time.time()
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        sync_all()
        h1 = time.time()
        ms_total = t0.elapsed_time(t1)
        if world > 1:
            tt = torch.tensor([ms_total], device=dev, dtype=torch.float64)
            tdist.all_reduce(tt, op=tdist.ReduceOp.MAX)
            ms_total = float(tt.item())
        # ---- the same K steps again with an event pair around every launch: each kernel's mean duration ----
        ev = {(k, M): [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
              for k in KS for M in MS}
        sync_all()
        for s in range(args.steps):
            step({key: ev[key][s] for key in ev})
        sync_all()
        per_launch, spread = {}, {}
        for key in ev:
            ts = sorted(e[0].elapsed_time(e[1]) for e in ev[key])
            per_launch[key] = sum(ts) / len(ts)
            spread[key] = (ts[int(0.1 * (len(ts) - 1))], ts[int(0.9 * (len(ts) - 1))])
        step_bytes = sum(packed_bytes(k) for k in KS for M in MS)
        res.update(value=world * step_bytes * args.steps / (ms_total * 1e-3) / 1e9, ms_total=ms_total,
                   per_launch=per_launch, spread=spread, launches=len(KS) * len(MS) * args.steps,
                   timed_window=(h0, h1))
        res["e2e"] = run_e2e(args, torch, tdist, tb, dev, stream, bufs, scales, geoms, xs, rot, world, sync_all)
        if rank == 0 or args.all_rows:
            timer = Timer(torch, dev, stream, max(args.steps, 20))
            res["rows"] = run_rows(torch, tb, inputs, dev, timer, l2, bufs, scales, geoms)
        res["clocks_all"] = clk.summary()
        res["clocks_timed"] = clk.summary(res["timed_window"])
    if world > 1:
        tdist.barrier()
        tdist.destroy_process_group()
    return res


def run_e2e(args, torch, tdist, tb, dev, stream, bufs, scales, geoms, xs, rot, world, sync_all):
    """The headline through the C ABI with host buffers: each launch is one trellis_matvec_axis1_host call, which
    queues the copy of its x from pinned host memory, the matvec and the transfer of its output back to pinned host
    memory, in order on its stream (pinned buffers are reached through their device mapping: a fetch kernel brings
    x in over the host link and the matvec stores its output straight into host memory).  Each (k, M) slot has its own host and device buffers; the arguments are
    prepared once (pointers, geometry, stream), as for the device-timed headline.

    `value` runs every call on the launching stream, so the matvecs run one after another as in the
    device-timed step, each behind its copies.  `two_streams` alternates the slots between two streams: one
    slot's copies then overlap the other stream's matvec, and matvecs of the two streams may also overlap one
    another, which the one-stream figure excludes."""
    lib = tb.load()
    slots = [(k, M) for k in KS for M in MS]
    x_host = {M: xs[M].cpu().pin_memory() for M in MS}
    o_host = {s: torch.empty((s[1], R), dtype=torch.bfloat16).pin_memory() for s in slots}
    x_dev = {s: torch.empty_like(xs[s[1]]) for s in slots}
    o_dev = {s: torch.empty((s[1], R), dtype=torch.bfloat16, device=dev) for s in slots}
    fn = lib.trellis_matvec_axis1_host

    def timed(streams):
        cargs = {}
        for j, (k, M) in enumerate(slots):  # the binding's checks once, then the prepared C arguments
            sp = streams[j % len(streams)]
            with torch.cuda.stream(sp):
                tb.matvec_axis1_host(bufs[k][0], scales[k], x_host[M], geoms[k], o_host[(k, M)], x_dev[(k, M)],
                                     o_dev[(k, M)])
            for i, b in enumerate(bufs[k]):
                cargs[(k, M, i)] = (b.data_ptr(), scales[k].data_ptr(), x_host[M].data_ptr(),
                                    o_host[(k, M)].data_ptr(), M, ctypes.byref(geoms[k].c()), x_dev[(k, M)].data_ptr(),
                                    o_dev[(k, M)].data_ptr(), sp.cuda_stream)

        def e2e_step():
            for (k, M) in slots:
                i = rot[k]
                rot[k] = (i + 1) % len(bufs[k])
                st = fn(*cargs[(k, M, i)])
                if st:
                    raise RuntimeError(f"trellis_matvec_axis1_host returned {st}")

        for _ in range(args.warmup):
            e2e_step()
        sync_all()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for sp in streams:
            if sp is not stream:
                sp.wait_event(a)
        for _ in range(args.steps):
            e2e_step()
        for sp in streams:
            if sp is not stream:
                stream.wait_stream(sp)
        b.record(stream)  # after the last output's copy to the host
        sync_all()
        ms = a.elapsed_time(b)
        if world > 1:
            tt = torch.tensor([ms], device=dev, dtype=torch.float64)
            tdist.all_reduce(tt, op=tdist.ReduceOp.MAX)
            ms = float(tt.item())
        return world * sum(packed_bytes(k) for k in KS for M in MS) * args.steps / (ms * 1e-3) / 1e9

    one = timed([stream])
    two = timed([torch.cuda.Stream(dev), torch.cuda.Stream(dev)])
    return {"value": one, "unit": "GB/s",
            "h2d_bytes_per_step": sum(M * C * 2 for k in KS for M in MS),
            "d2h_bytes_per_step": sum(M * R * 2 for k in KS for M in MS),
            "call": "trellis_matvec_axis1_host (one C call per launch: x in, matvec, out back), all on one stream",
            "two_streams": {"value": two, "unit": "GB/s",
                            "how": "the same calls alternating between two streams: copies overlap the other "
                                   "stream's matvec, and the two streams' matvecs may overlap"}}


def run_rows(torch, tb, inputs, dev, timer, l2, bufs, scales, geoms):
    """Every other row of the hot path at its full size (see the module docstring).  Each entry: the row's
    kind, k, M, mean and p10/p90 launch time, and its algorithmic bytes (matvecs, expand, floors) or FLOPs
    (prefill); fractions are added by main() from the measured peaks."""
    rows = []

    def code_set(per_launch_bytes, k, seed, mult=1):
        nrot = int(2 * l2 // per_launch_bytes) + 2
        return [_dev_words(inputs.random_words(seed + 37 * i + k, (R, C * k // 32)), dev) for i in range(nrot * mult)]

    sc = _dev_f16(inputs.uniform_f16(inputs.SEED_SCALES, (R,)), dev)

    # ---- config 3: fused gate/up SwiGLU, two [17408, 5120] matrices ----
    for k in (2, 3):
        cs = code_set(2 * packed_bytes(k), k, 9000, 2)
        g = tb.Geometry(k, L, T, 1, R, C)
        for M in MS:
            x = _dev_bf16(inputs.normal_bf16(inputs.SEED_X + M, (M, C)), dev)
            o = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
            t = timer(lambda i: tb.gateup_swiglu(cs[2 * i], sc, cs[2 * i + 1], sc, x, g, o), len(cs) // 2)
            rows.append({"kind": "gateup", "config": 3, "k": k, "M": M, **t,
                         "bytes": 2 * packed_bytes(k) + 4 * R + 2 * M * C + 2 * M * R})
        del cs
    # ---- config 4: axis-0 down projection, stored W^T [17408 in, 5120 out] ----
    for k in (2, 3):
        cs = code_set(packed_bytes(k), k, 9500)
        g = tb.Geometry(k, L, T, 0, R, C)
        for M in MS:
            x = _dev_bf16(inputs.normal_bf16(inputs.SEED_X + 10 + M, (M, R), 0.5), dev)
            o = torch.empty((M, C), dtype=torch.bfloat16, device=dev)
            ws = tb.new_workspace(M, g, dev)
            t = timer(lambda i: tb.matvec_axis0(cs[i], sc, x, g, ws, o), len(cs))
            rows.append({"kind": "axis0", "config": 4, "k": k, "M": M, **t,
                         "bytes": packed_bytes(k) + 2 * R + 2 * M * R + 2 * M * C})
        del cs
    # ---- expand to bf16 (the transient of the comparator) ----
    o = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
    for k in KS:
        g = geoms[k]
        t = timer(lambda i: tb.expand_bf16(bufs[k][i], scales[k], g, o), len(bufs[k]))
        rows.append({"kind": "expand", "config": 2, "k": k, "M": 0, **t, "bytes": packed_bytes(k) + 2 * R + 2 * R * C})
    del o
    # ---- load-only floors of the packed stream (the M = 1 pattern, and fully coalesced) ----
    fout = torch.empty(R, dtype=torch.int32, device=dev)
    for k in KS:
        for coal in (False, True):
            t = timer(lambda i: tb.load_floor(bufs[k][i], geoms[k], fout, coalesced=coal), len(bufs[k]))
            rows.append({"kind": "load_floor_coalesced" if coal else "load_floor", "config": 2, "k": k, "M": 0, **t,
                         "bytes": packed_bytes(k) + 4 * R})
    # ---- config 5: tensor-core prefill (axis 1, k = 2) and expand + cuBLAS ----
    k = 2
    g = tb.Geometry(k, L, T, 1, R, C)
    wtmp = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
    cs = code_set(packed_bytes(k), k, 5000)
    for M in PREFILL_M:
        x = _dev_bf16(inputs.normal_bf16(inputs.SEED_X + 5000 + M, (M, C)), dev)
        o = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
        t = timer(lambda i: tb.gemm_prefill(cs[i], sc, x, g, o), len(cs))
        tc = timer(lambda i: torch.matmul(x, tb.expand_bf16(cs[i], sc, g, wtmp).t()), len(cs))
        rows.append({"kind": "prefill", "config": 5 if M >= 32 else None, "k": k, "M": M, **t,
                     "flops": 2.0 * M * R * C,
                     "comparator": {"what": "trellis_expand_bf16 + torch.matmul (cuBLAS)", **tc}})
    del cs
    # ---- axis-0 prefill (the down projection for M > 4), k = 3, stored W^T [17408 in, 5120 out] ----
    k = 3
    g0 = tb.Geometry(k, L, T, 0, R, C)
    cs = code_set(packed_bytes(k), k, 6000)
    for M in PREFILL0_M:
        x = _dev_bf16(inputs.normal_bf16(inputs.SEED_X + 6000 + M, (M, R), 0.5), dev)
        o = torch.empty((M, C), dtype=torch.bfloat16, device=dev)
        t = timer(lambda i: tb.gemm_prefill(cs[i], sc, x, g0, o), len(cs))
        tc = timer(lambda i: torch.matmul(x, tb.expand_bf16(cs[i], sc, g0, wtmp)), len(cs))
        rows.append({"kind": "prefill_axis0", "config": 5, "k": k, "M": M, **t, "flops": 2.0 * M * R * C,
                     "comparator": {"what": "trellis_expand_bf16 + torch.matmul (cuBLAS)", **tc}})
    del cs, wtmp
    # ---- decode MLP block (gate/up SwiGLU + down) replayed as CUDA graphs ----
    for ku, kd in ((2, 2), (3, 3)):
        g_up, g_dn = tb.Geometry(ku, L, T, 1, R, C), tb.Geometry(kd, L, T, 0, R, C)
        wsets = [[_dev_words(inputs.random_words(7000 + 10 * i + j, (R, C * (ku if j < 2 else kd) // 32)), dev)
                  for j in range(3)] for i in range(3)]
        for M in MS:
            graphs = [tb.MlpDecodeGraph(w[0], sc, w[1], sc, w[2], sc, g_up, g_dn, M) for w in wsets]
            for gr in graphs:
                gr.x.copy_(_dev_bf16(inputs.normal_bf16(inputs.SEED_X, (M, C)), dev))
            t = timer(lambda i: graphs[i].replay(), len(graphs))
            rows.append({"kind": "mlp_graph", "config": 3, "k": ku, "k_down": kd, "M": M, **t,
                         "bytes": 2 * packed_bytes(ku) + packed_bytes(kd)})
            del graphs
        del wsets
    return rows


def cpu_baseline(seconds: float = 12.0):
    """The oracle as it stands (one host core) on a bounded sample of rows of
    the same twelve (k, M) launches; GB/s of the sampled rows' packed bytes."""
    import oracle
    from trellis_coded_weight_gb300 import inputs
    oracle.build()
    data = {k: inputs.make_linear(R, C, k, 4, seed_codes=inputs.SEED_CODES + k) for k in KS}
    rows_per = 8
    t = time.perf_counter()
    for k in KS:  # calibrate on a tiny sample
        oracle.matvec_axis1(data[k][0], data[k][1], data[k][2][:1], k, L, T, rows=np.arange(rows_per))
    per_row = (time.perf_counter() - t) / (rows_per * len(KS))
    n = max(8, int(seconds / (per_row * len(KS) * len(MS))))
    n = min(n, R)
    rng = np.random.default_rng(1)
    idx = np.sort(rng.choice(R, n, replace=False)).astype(np.int64)
    nbytes = 0
    t = time.perf_counter()
    for k in KS:
        for M in MS:
            oracle.matvec_axis1(data[k][0], data[k][1], data[k][2][:M], k, L, T, rows=idx)
            nbytes += n * C * k // 8
    dt = time.perf_counter() - t
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} random rows (of {R}) of each of the 12 (k, M) matvecs, {dt:.1f} s on one core",
            "per_row_s": dt / (n * len(KS) * len(MS))}


def cpu_baseline_prefill(seconds: float = 10.0):
    """The oracle's prefill (bf16 expand weights, double sums) on one host core for a bounded random sample of
    output features of the M = 2048 prefill; TFLOP/s of the sampled outputs (2 * M * C per feature)."""
    import oracle
    from trellis_coded_weight_gb300 import inputs
    oracle.build()
    M = PREFILL_M[-1]
    codes, scales, _ = inputs.make_linear(R, C, 2, 1, seed_codes=inputs.SEED_CODES + 5000)
    x = inputs.normal_bf16(inputs.SEED_X + 5000 + M, (M, C))
    t = time.perf_counter()
    oracle.prefill(codes, scales, x, 2, L, T, rows=np.arange(2))
    per = (time.perf_counter() - t) / 2
    n = int(max(4, min(R, seconds / max(per, 1e-6))))
    idx = np.sort(np.random.default_rng(2).choice(R, n, replace=False)).astype(np.int64)
    t = time.perf_counter()
    oracle.prefill(codes, scales, x, 2, L, T, rows=idx)
    dt = time.perf_counter() - t
    return {"value": 2.0 * M * C * n / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} random output features (of {R}) x all {M} tokens of the k=2 prefill, {dt:.1f} s on one core"}


_POOL_DATA = None


def _pool_init():
    """Worker set-up (spawned process): the oracle library and the seeded inputs of each k."""
    global _POOL_DATA
    import oracle
    from trellis_coded_weight_gb300 import inputs
    oracle.build()
    _POOL_DATA = {k: inputs.make_linear(R, C, k, 4, seed_codes=inputs.SEED_CODES + k) for k in KS}


def _pool_rows(task):
    import oracle
    k, M, lo, hi = task
    codes, scales, x = _POOL_DATA[k]
    oracle.matvec_axis1(codes, scales, x[:M], k, L, T, rows=np.arange(lo, hi, dtype=np.int64))
    return (hi - lo) * C * k // 8


def cpu_baseline_all_cores(per_row_s: float, seconds: float = 8.0):
    """The same oracle on every host core: a spawn-started process pool, each task one row range of one
    of the 12 (k, M) matvecs (the oracle itself is the single-threaded code, unchanged).  per_row_s is
    the single-core cost of one row (averaged over the 12 launches), which sizes the row ranges."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    chunk = int(seconds / (len(KS) * len(MS) * max(per_row_s, 1e-7)))
    chunk = max(8, min(chunk, R // cores))
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_pool_init) as pool:
        pool.map(_pool_rows, [(2, 1, i, i + 1) for i in range(cores)])  # every worker is set up
        tasks = [(k, M, w * chunk, (w + 1) * chunk) for k in KS for M in MS for w in range(cores)]
        t = time.perf_counter()
        nbytes = sum(pool.map(_pool_rows, tasks, chunksize=1))
        dt = time.perf_counter() - t
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"rows 0..{cores * chunk} of each of the 12 (k, M) matvecs, {dt:.1f} s on {cores} cores"}


def run_reference(args):
    """Reference arm: the oracle, timed on host cores, same metric and config."""
    import oracle
    from trellis_coded_weight_gb300 import inputs
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    oracle.build()
    data = {k: inputs.make_linear(R, C, k, 4, seed_codes=inputs.SEED_CODES + k) for k in KS}
    rows = 96  # rows per launch: one step is about 0.5 s of one core
    idx = np.arange(rows, dtype=np.int64)

    def step():
        for k in KS:
            for M in MS:
                oracle.matvec_axis1(data[k][0], data[k][1], data[k][2][:M], k, L, T, rows=idx)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    nbytes = sum(rows * C * k // 8 for k in KS for M in MS) * args.steps
    v = nbytes / dt / 1e9
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded SplitMix64)", "config": workload_desc(),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{rows} rows (of {R}) of each of the 12 (k, M) matvecs per step"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_single(kind: str, k: str, M: str):
    """Four launches of one kernel on the full-size workload (for ncu: -s 3 -c 1)."""
    import torch
    from trellis_coded_weight_gb300 import binding as tb
    from trellis_coded_weight_gb300 import build as tbuild
    from trellis_coded_weight_gb300 import inputs
    k, M = int(k), int(M)
    dev = torch.device("cuda", 0)
    tbuild.build()
    tb.load()
    codes = _dev_words(inputs.random_words(inputs.SEED_CODES, (R, C * k // 32)), dev)
    codes2 = _dev_words(inputs.random_words(inputs.SEED_UP, (R, C * k // 32)), dev)
    sc = _dev_f16(inputs.uniform_f16(inputs.SEED_SCALES, (R,)), dev)
    g1, g0 = tb.Geometry(k, L, T, 1, R, C), tb.Geometry(k, L, T, 0, R, C)
    if kind == "axis1":
        x = _dev_bf16(inputs.normal_bf16(inputs.SEED_X, (M, C)), dev)
        fn = lambda: tb.matvec_axis1(codes, sc, x, g1)
    elif kind == "gateup":
        x = _dev_bf16(inputs.normal_bf16(inputs.SEED_X, (M, C)), dev)
        fn = lambda: tb.gateup_swiglu(codes, sc, codes2, sc, x, g1)
    elif kind == "axis0":
        x = _dev_bf16(inputs.normal_bf16(inputs.SEED_X, (M, R), 0.5), dev)
        ws = tb.new_workspace(M, g0, dev)
        fn = lambda: tb.matvec_axis0(codes, sc, x, g0, ws)
    elif kind == "expand":
        fn = lambda: tb.expand_bf16(codes, sc, g1)
    elif kind == "prefill":
        x = _dev_bf16(inputs.normal_bf16(inputs.SEED_X, (M, C)), dev)
        fn = lambda: tb.gemm_prefill(codes, sc, x, g1)
    elif kind == "prefill0":  # axis-0 prefill: the stored W^T [R in][C out]
        x = _dev_bf16(inputs.normal_bf16(inputs.SEED_X, (M, R), 0.5), dev)
        fn = lambda: tb.gemm_prefill(codes, sc, x, g0)
    elif kind in ("floor", "floor_rows"):
        fn = lambda: tb.load_floor(codes, g1, coalesced=kind == "floor_rows")
    else:
        raise SystemExit(f"unknown kind {kind}")
    for _ in range(4):
        fn()
    torch.cuda.synchronize(dev)
    print(json.dumps({"single": kind, "k": k, "M": M, "device_error": tb.device_error()}))


def kernel_source_hash(*names: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in names + ("common.cuh",):
        with open(os.path.join(ROOT, "trellis_coded_weight_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_profile(key: str):
    """A committed ncu figure (DRAM bytes and instructions per launch) of a kernel, or None when the kernel's
    source changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f).get(key)
        if d and d.get("source_hash") == kernel_source_hash(*d["sources"]):
            return d
    except Exception:
        pass
    return None


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--all-rows", action="store_true", help="under torchrun, time the other rows on every rank")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--single", nargs=3, metavar=("KIND", "K", "M"),
                    help="profiling aid: run 4 launches of one kernel at full size and exit "
                         "(KIND: axis1, gateup, axis0, expand, prefill, prefill0, floor, floor_rows)")
    args = ap.parse_args()
    if args.single:
        run_single(*args.single)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.impl == "reference":
        res = run_reference(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    res = run_gpu(args)
    if res["rank"] != 0:
        return
    peaks, peak_src = load_peaks()
    world = res["world"]
    hbm = float(peaks["hbm_gbs"])
    bf16_peak = float(peaks["bf16_tflops"])
    per = res["per_launch"]
    alg = {(k, M): packed_bytes(k) + 2 * R + 2 * M * C + 2 * M * R for k in KS for M in MS}

    # roofline of the dominant kernel: the axis-1 matvec (every timed launch is one).  Bound by HBM in the
    # metric's terms: algorithmic bytes per launch over the mean launch time against the measured copy rate.
    # The mean launch time is the timed region's events over its launches (back-to-back, as the step runs
    # them); the second pass's event pair around every launch also gives it, but those events stop each
    # launch from overlapping the previous one's end (programmatic dependent launch), so that figure is
    # reported beside it.
    step_s = res["ms_total"] * 1e-3 / args.steps  # one rank's step (each rank runs the same step)
    achieved = sum(alg.values()) / step_s / 1e9
    achieved_events = sum(alg.values()) / (sum(per.values()) * 1e-3) / 1e9
    prof = [measured_profile(f"axis1_k{k}_M{M}") for k in KS for M in MS]
    traffic = (sum(p["dram_bytes_per_launch"] for p in prof) / len(prof)) if all(prof) else None
    floors = {r["kind"] + f"_k{r['k']}": packed_bytes(r["k"]) / (r["us"] * 1e-6) / 1e9
              for r in res.get("rows", []) if r["kind"].startswith("load_floor")}
    roofline = {"kernel": "trellis_matvec_axis1 (mv1_kernel at M = 1, mvtc_kernel at M >= 2)", "bound": "hbm",
                "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "mean_launch_us": step_s / len(alg) * 1e6,
                "achieved_per_launch_events": {"value": achieved_events, "frac": achieved_events / hbm,
                                               "mean_launch_us": sum(per.values()) / len(per) * 1e3},
                "peak_source": f"{peak_src} hbm_gbs (copy)",
                "algorithmic_bytes_per_launch": sum(alg.values()) / len(alg),
                "traffic": traffic, "load_floor_GBps": floors}
    if all(prof):
        # issue view: the warp-instructions ncu counted per launch, over the mean launch time, against one
        # instruction per cycle per SM sub-partition at the maximum SM clock
        import torch
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        mhz = float(res["clocks_all"].get("sm_max_mhz") or 2070.0)
        inst = sum(p["warp_instructions_per_launch"] for p in prof)
        ach = inst / step_s / 1e12
        peak_i = sms * 4 * mhz * 1e6 / 1e12
        roofline["issue"] = {"achieved": ach, "peak": peak_i, "unit": "T warp-instructions/s", "frac": ach / peak_i,
                             "peak_source": f"derived: {sms} SMs x 4 schedulers x 1 instruction/clock x {mhz:.0f} MHz",
                             "instructions_per_weight": inst * 32 / (R * C * len(alg)),
                             "source": "ncu smsp__inst_executed.sum, profiles/traffic.json"}
    breakdown = [{"kind": "axis1", "config": 2, "k": k, "M": M, "us": per[(k, M)] * 1e3,
                  "us_p10_p90": [res["spread"][(k, M)][0] * 1e3, res["spread"][(k, M)][1] * 1e3],
                  "bytes": alg[(k, M)], "GBps": alg[(k, M)] / (per[(k, M)] * 1e-3) / 1e9,
                  "packed_GBps": packed_bytes(k) / (per[(k, M)] * 1e-3) / 1e9,
                  "frac_hbm": alg[(k, M)] / (per[(k, M)] * 1e-3) / 1e9 / hbm} for k in KS for M in MS]
    prefill = None
    for r in res.get("rows", []):
        if "bytes" in r:
            r["GBps"] = r["bytes"] / (r["us"] * 1e-6) / 1e9
            r["frac_hbm"] = r["GBps"] / hbm
            if r["kind"] in ("gateup", "axis0", "mlp_graph"):
                packed = (2 * packed_bytes(r["k"]) if r["kind"] == "gateup" else packed_bytes(r["k"]))
                if r["kind"] == "mlp_graph":
                    packed = 2 * packed_bytes(r["k"]) + packed_bytes(r["k_down"])
                r["packed_GBps"] = packed / (r["us"] * 1e-6) / 1e9
        else:
            r["TFLOPs"] = r["flops"] / (r["us"] * 1e-6) / 1e12
            r["frac_bf16"] = r["TFLOPs"] / bf16_peak
            r["comparator"]["TFLOPs"] = r["flops"] / (r["comparator"]["us"] * 1e-6) / 1e12
            if r["kind"] == "prefill" and r["M"] == PREFILL_M[-1]:
                prefill = {"M": r["M"], "k": r["k"], "rows": R, "cols": C, "ms": r["us"] * 1e-3, "tflops": r["TFLOPs"],
                           "frac": r["frac_bf16"], "peak": bf16_peak, "peak_source": f"{peak_src} bf16_tflops (burst)",
                           "comparator": {"what": r["comparator"]["what"], "ms": r["comparator"]["us"] * 1e-3,
                                          "tflops": r["comparator"]["TFLOPs"]}}
        breakdown.append(r)
    clocks = dict(res["clocks_all"])
    clocks["window"] = "from the first warm-up step to the last timed row"
    clocks["timed_region"] = res["clocks_timed"]
    line = {
        "metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_total"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded SplitMix64 code words, fp16 scales U[0.005,0.02], bf16 x ~ N(0,1)",
        "config": workload_desc(), "frac_hbm": res["value"] / world / hbm,
        "roofline": roofline, "e2e": res["e2e"], "gpu_launches": res["launches"], "clocks": clocks,
        "prefill": prefill, "breakdown": breakdown,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
        try:
            line["cpu_baseline"]["all_cores"] = cpu_baseline_all_cores(line["cpu_baseline"].pop("per_row_s"))
        except Exception as e:  # the single-core figure stands on its own
            line["cpu_baseline"]["all_cores"] = {"unavailable": str(e)[:200]}
        try:
            line["cpu_baseline"]["prefill"] = cpu_baseline_prefill()
        except Exception as e:
            line["cpu_baseline"]["prefill"] = {"unavailable": str(e)[:200]}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
