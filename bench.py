"""Benchmark of the scaled-FP8 GEMM path on GB300.

Default workload (one "step"): the Float8 linear forward + backward with
per-tensor current scaling -- x[8192,2048] (E4M3), W[2048,2048] (E4M3),
grad_out[8192,2048] (E5M2), bf16 in and out: current scaling of x, g and W
in one launch (amax, scale and row-major codes of each, the reduction of one
tensor overlapped with the cast of the previous), then the three GEMMs
y = x W^T, dx = g W, dW = g^T x in one grouped launch that reads the codes
K-major or MN-major as each GEMM needs.

Printed: one JSON line with the headline metric (FP8 scaled-GEMM TFLOP/s
including quantization), the GEMM roofline against the dense FP8 peak, the
quantize kernels' HBM roofline, an end-to-end number through the public API
with host buffers, the CPU oracle timed on a bounded sample, and the clocks
sampled during the timed region.  ``--impl reference`` times the CPU oracle
on the same workload instead.  ``--workload`` selects another configuration.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--no-extras]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

L2_FLUSH_BYTES = 512 << 20  # > the 129 MB L2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_%d_" % os.getpid(), suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # median over the samples taken under load (clock above idle floor)
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- timing kit --

class StepTimer:
    """Per-launch CUDA events on the launching stream across the timed steps."""

    def __init__(self):
        self.records = []  # (label, start_event, end_event)
        self.steps = []    # (start_event, end_event)

    def launch(self, label, fn, stream):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        self.records.append((label, s, e))

    def per_label_ms(self):
        out = {}
        for label, s, e in self.records:
            out.setdefault(label, []).append(s.elapsed_time(e))
        return out

    def step_ms(self):
        return [s.elapsed_time(e) for s, e in self.steps]


# -------------------------------------------------------------- workloads --

def pinned(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().pin_memory()


class Float8Linear:
    """Float8 linear forward + backward, per-tensor current scaling.

    Each tensor is quantized once, to row-major codes; the GEMMs read them in
    the layout they need: y = x W^T takes x_q and W_q K-major; dx = g W takes
    g_q K-major and W_q MN-major; dW = g^T x takes g_q and x_q MN-major (no
    transposed copies are written)."""

    name = "float8_linear_fwd_bwd"

    def __init__(self, dev, tokens=8192, d_in=2048, d_out=2048):
        import fp8_quantized_gemm_gb300 as F
        self.F = F
        self.T, self.din, self.dout = tokens, d_in, d_out
        x, w, g = workloads.float8_linear(tokens=tokens, d_in=d_in, d_out=d_out)
        self.host_in = [pinned(x), pinned(w), pinned(g)]
        self.x, self.w, self.g = (t.to(dev) for t in self.host_in)
        u8 = dict(dtype=torch.uint8, device=dev)
        T, di, do = tokens, d_in, d_out
        self.xq = torch.empty((T, di), **u8)
        self.wq = torch.empty((do, di), **u8)
        self.gq = torch.empty((T, do), **u8)
        self.amax = torch.empty(3, device=dev)
        self.scale = torch.empty(3, device=dev)
        self.sync = torch.zeros(F.QUANT_SYNC_WORDS, dtype=torch.int32, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.y, self.dx, self.dw = torch.empty((T, do), **bf), torch.empty((T, di), **bf), \
            torch.empty((do, di), **bf)
        self.outputs = [self.y, self.dx, self.dw]
        self.host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in self.outputs]
        self.flops = 3 * 2.0 * T * di * do
        n_x, n_w, n_g = T * di, do * di, T * do
        self.n_elems = n_x + n_w + n_g
        # algorithmic HBM bytes per step: current scaling of x, g and W reads
        # each input once (2 B/elem) and writes its codes (1 B/elem)
        self.bytes = {"quantize": 3.0 * self.n_elems}
        # x, g and W in one launch, in that order (the small W last: while one
        # tensor is cast the next is reduced, so the last one is the tail)
        s = self.scale
        self.items = [F.quant_item(self.x, F.E4M3, self.xq, s[0:1], self.amax[0:1]),
                      F.quant_item(self.g, F.E5M2, self.gq, s[2:3], self.amax[2:3]),
                      F.quant_item(self.w, F.E4M3, self.wq, s[1:2], self.amax[1:2])]
        # the three GEMMs (y = x W^T, dx = g W, dW = g^T x) as one grouped call
        MN = F.MN_MAJOR
        self.problems = [
            F.gemm_problem(self.xq, F.E4M3, self.wq, F.E4M3, s[0:1], s[1:2], self.y),
            F.gemm_problem(self.gq, F.E5M2, self.wq, F.E4M3, s[2:3], s[1:2], self.dx,
                           b_layout=MN),
            F.gemm_problem(self.gq, F.E5M2, self.xq, F.E4M3, s[2:3], s[0:1], self.dw,
                           a_layout=MN, b_layout=MN),
        ]
        self.h2d = sum(t.numel() * t.element_size() for t in self.host_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.outputs)

    def launches(self):
        F = self.F
        return [
            ("quantize", lambda: F.fp8_quantize_tensors(self.items, self.sync)),
            ("gemm", lambda: F.fp8_gemm_tensor_grouped(self.problems)),
        ]

    def upload(self, stream):
        for h, d in zip(self.host_in, (self.x, self.w, self.g)):
            d.copy_(h, non_blocking=True)

    def download(self, stream):
        for d, h in zip(self.outputs, self.host_out):
            h.copy_(d, non_blocking=True)

    def io_set(self):
        """A second set of device inputs and outputs with its own launch list
        (the codes, scales and scratch are shared: steps compute one after
        another on one stream), for overlapping one step's copies with the
        neighbouring steps' compute."""
        F, dev = self.F, self.x.device
        st = Float8Linear.__new__(Float8Linear)
        st.F, st.host_in, st.host_out = F, self.host_in, self.host_out
        st.x, st.w, st.g = (torch.empty_like(t) for t in (self.x, self.w, self.g))
        st.y, st.dx, st.dw = (torch.empty_like(t) for t in (self.y, self.dx, self.dw))
        st.outputs = [st.y, st.dx, st.dw]
        s, MN = self.scale, F.MN_MAJOR
        st.sync = self.sync
        st.items = [F.quant_item(st.x, F.E4M3, self.xq, s[0:1], self.amax[0:1]),
                    F.quant_item(st.g, F.E5M2, self.gq, s[2:3], self.amax[2:3]),
                    F.quant_item(st.w, F.E4M3, self.wq, s[1:2], self.amax[1:2])]
        st.problems = [
            F.gemm_problem(self.xq, F.E4M3, self.wq, F.E4M3, s[0:1], s[1:2], st.y),
            F.gemm_problem(self.gq, F.E5M2, self.wq, F.E4M3, s[2:3], s[1:2], st.dx, b_layout=MN),
            F.gemm_problem(self.gq, F.E5M2, self.xq, F.E4M3, s[2:3], s[0:1], st.dw,
                           a_layout=MN, b_layout=MN),
        ]
        return st

    # ---- CPU oracle on a bounded sample: the first `rows` token rows
    def oracle_sample(self, rows):
        from oracle import gemm as OG
        from oracle import quantize as OQ
        x, w, g = self.host_in
        xs, gs, wf = x[:rows].float().numpy(), g[:rows].float().numpy(), w.float().numpy()
        t0 = time.perf_counter()
        qx, sx = OQ.quantize_tensor(xs, "e4m3")
        qw, sw = OQ.quantize_tensor(wf, "e4m3")
        qg, sg = OQ.quantize_tensor(gs, "e5m2")
        xd = OG.dequant_operand(qx, "e4m3", sx)
        wd = OG.dequant_operand(qw, "e4m3", sw)
        gd = OG.dequant_operand(qg, "e5m2", sg)
        OG.gemm(xd, wd)            # y  = x W^T
        OG.gemm(gd, wd.T)          # dx = g W
        OG.gemm(gd.T, xd.T)        # dW = g^T x (partial over the sampled rows)
        dt = time.perf_counter() - t0
        flops = 3 * 2.0 * rows * self.din * self.dout
        return flops, dt, "first %d of %d token rows (x, g), full W; 3 quantizes + 3 GEMMs" % (
            rows, self.T)


# ----------------------------------------------------------- distributed --

def setup_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return torch.device("cuda", torch.cuda.current_device()), rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """Largest value over all ranks (the timing every rank reports is the
    slowest rank's)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, steps: int, rank_total_ms: float, world: int) -> float:
    """Whole-job throughput: the units every rank processed in `steps` steps,
    over the slowest rank's time (per second)."""
    slowest_ms = max_over_ranks(rank_total_ms, world)
    return units_per_rank * steps * world / (slowest_ms / 1e3)


def source_digest(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    source has not changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh).get(kernel)
    if not rec:
        return None
    if rec.get("source_digest") != source_digest(rec["sources"]):
        return None
    return rec["dram_bytes_per_launch"]


# ------------------------------------------------------------- our arm --

def time_workload(wl, steps, warmup, world, flush, stream):
    launches = wl.launches()
    for _ in range(warmup):
        for _, fn in launches:
            fn()
    torch.cuda.synchronize()
    timer = StepTimer()
    barrier(world)
    torch.cuda.synchronize()
    for _ in range(steps):
        flush.zero_()  # write 512 MiB: evicts the 129 MB L2 between steps
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for label, fn in launches:
            timer.launch(label, fn, stream)
        e.record(stream)
        timer.steps.append((s, e))
    torch.cuda.synchronize()
    barrier(world)
    return timer, len(launches)


SPIN_CYCLES = 400_000  # ~0.2 ms at 2 GHz


def time_isolated(wl, reps, flush, stream):
    """Device time of each launch in step order: L2 is flushed once at the
    start of every pass (as between timed steps), and a spin kernel that
    touches no memory is queued before every launch so the host enqueues the
    launch while the GPU spins; the events then bracket the kernel alone, with
    the cache state the step itself leaves (e.g. a GEMM reads the codes its
    quantize pass just wrote)."""
    per = {}
    launches = wl.launches()
    for _ in range(reps):
        flush.zero_()
        for label, fn in launches:
            torch.cuda._sleep(SPIN_CYCLES)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            per.setdefault(label, []).append((s, e))
    torch.cuda.synchronize()
    return {k: [s.elapsed_time(e) for s, e in v] for k, v in per.items()}


def time_graph(wl, steps, world, flush):
    """The same step captured once as a CUDA graph and replayed: the kernels
    and their order are unchanged, the host launch gaps between them go."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _, fn in wl.launches():  # warm the capture stream
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        if hasattr(wl, "capture_branches"):
            wl.capture_branches()
        else:
            for _, fn in wl.launches():
                fn()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    times = []
    barrier(world)
    torch.cuda.synchronize()
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        graph.replay()
        e.record(stream)
        times.append((s, e))
    torch.cuda.synchronize()
    barrier(world)
    return [s.elapsed_time(e) for s, e in times]


def time_e2e_pipelined(wl, steps, stream):
    """End to end with each step's H2D copy and D2H read inside the timed
    region, steps overlapped: step i+1's inputs are copied in (copy stream 1)
    while step i computes, and step i's outputs are read back (copy stream 2)
    while step i+1 computes -- two sets of device inputs and outputs
    alternate.  Returns the mean time per step over `steps` steps."""
    sets = [wl, wl.io_set()]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    comp = stream
    for st in sets:  # warm both sets once
        st.upload(comp)
        for _, fn in st.launches():
            fn()
        st.download(comp)
    torch.cuda.synchronize()
    done_comp, done_out = [None, None], [None, None]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    s_in.wait_stream(comp)
    s_out.wait_stream(comp)
    for i in range(steps):
        b = i % 2
        st = sets[b]
        with torch.cuda.stream(s_in):
            if done_comp[b] is not None:
                s_in.wait_event(done_comp[b])   # the previous user of set b has read it
            st.upload(s_in)
            arrived = torch.cuda.Event()
            arrived.record(s_in)
        comp.wait_event(arrived)
        if done_out[b] is not None:
            comp.wait_event(done_out[b])        # set b's outputs have been read back
        for _, fn in st.launches():
            fn()
        done_comp[b] = torch.cuda.Event()
        done_comp[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done_comp[b])
            st.download(s_out)
            done_out[b] = torch.cuda.Event()
            done_out[b].record(s_out)
    comp.wait_stream(s_out)
    end.record(comp)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def time_e2e(wl, steps, flush, stream):
    launches = wl.launches()
    times = []
    for _ in range(steps):
        flush.zero_()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        wl.upload(stream)
        for _, fn in launches:
            fn()
        wl.download(stream)
        e.record(stream)
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e))
    return times


def cpu_baseline(wl, rows, min_seconds=10.0, max_reps=8):
    flops, dt, reps = 0.0, 0.0, 0
    while reps < max_reps and (dt < min_seconds or reps == 0):
        f, d, sample = wl.oracle_sample(rows)
        flops, dt, reps = flops + f, dt + d, reps + 1
    sample = "%s; %d repetition(s)" % (sample, reps)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": sample, "seconds": round(dt, 3)}


def same_flush_copy_gbs(nbytes, flush, stream, reps=10):
    """A plain device copy moving `nbytes` (half read, half written) after the
    same L2 flush as the timed launches: what a pure stream of that much
    traffic reaches under the flush protocol (the flush leaves L2 full of
    dirty lines, which the next kernel's traffic has to evict)."""
    src = torch.empty(nbytes // 2, dtype=torch.uint8, device=flush.device)
    dst = torch.empty_like(src)
    per, _ = time_launches([("copy", lambda: dst.copy_(src))], reps, flush, stream)
    return nbytes / (per["copy"] / 1e3) / 1e9


def roofline_entry(bound, achieved, peak, unit, traffic, note):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": note}


def run_ours(args):
    import fp8_quantized_gemm_gb300 as F
    peaks = load_peaks()
    dev, rank, world = setup_dist()
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    wl = Float8Linear(dev)
    with ClockSampler(dev.index) as clk:
        timer, n_launch = time_workload(wl, args.steps, args.warmup, world, flush, stream)
    rc, where = F.fp8_get_last_device_error()
    if rc != 0:
        raise RuntimeError("device error %d (where %d) during the timed region" % (rc, where))
    step_ms = timer.step_ms()
    eager_total_ms = max_over_ranks(sum(step_ms), world)
    eager_value = job_throughput(wl.flops, args.steps, sum(step_ms), world) / 1e12
    if args.eager:
        total_ms, value = eager_total_ms, eager_value
    else:
        with ClockSampler(dev.index) as clk:
            graph_ms = time_graph(wl, args.steps, world, flush)
        total_ms = max_over_ranks(sum(graph_ms), world)
        value = job_throughput(wl.flops, args.steps, sum(graph_ms), world) / 1e12
    reps = 10
    per = time_isolated(wl, reps, flush, stream)
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # dense FP8 = 2 x bf16 (nominal ratio)
    # algorithmic work of a step over the per-step device time of each kind
    gemm_tflops = wl.flops / (sum(per["gemm"]) / reps / 1e3) / 1e12
    q_gbs = wl.bytes["quantize"] / (sum(per["quantize"]) / reps / 1e3) / 1e9
    copy_gbs = same_flush_copy_gbs(int(wl.bytes["quantize"]), flush, stream)
    src = "MEASURED_PEAKS.json (%s)" % peaks["source"]
    line = {
        "metric": "FP8 scaled-GEMM TFLOP/s incl. quantize, % of FP8 peak; quantize GB/s % HBM",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8 e4m3/e5m2, fp32 accumulate", "data": "synthetic",
        "config": {"workload": wl.name, "tokens": wl.T, "d_in": wl.din, "d_out": wl.dout,
                   "scaling": "per-tensor current", "inputs": "bf16, seeded (workloads.py)",
                   "l2": "flushed between timed steps (512 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "fraction_of_fp8_peak": round(value / fp8_peak, 4),
        "roofline": roofline_entry("tensor", gemm_tflops, fp8_peak, "TFLOP/s",
                                   recorded_traffic("gemm_pair_grouped"),
                                   "dense FP8 = 2 x measured bf16 burst (%s)" % src),
        "quantize_roofline": dict(
            roofline_entry("hbm", q_gbs, peaks["hbm_gbs"], "GB/s",
                           recorded_traffic("quantize_multi"), "measured HBM copy (%s)" % src),
            same_flush_copy_gbs=round(copy_gbs, 1), frac_of_same_flush_copy=round(q_gbs / copy_gbs, 4)),
        "launch": "eager (one API call per kernel)" if args.eager else
                  "CUDA graph of the step's API calls, replayed",
        "eager": {"value": round(eager_value, 2), "ms_per_step": round(eager_total_ms / args.steps, 4)},
        "kernel_ms": {k: round(sum(v) / len(v), 4) for k, v in per.items()},
        "kernel_ms_note": "mean per launch: quantize is one launch for x, g and W (amax, "
                          "scale and codes of each), gemm one grouped launch of the three GEMMs",
        "kernel_timing": "each launch bracketed by CUDA events in step order, L2 flushed per "
                         "step, a memory-free spin kernel queued before each launch",
        "gpu_launches": n_launch * args.steps,
        "clocks": clk.summary(),
    }
    e2e_steps = max(3, min(args.steps, 50))
    if hasattr(wl, "io_set"):
        e2e_ms = max_over_ranks(time_e2e_pipelined(wl, e2e_steps, stream), world)
        how = ("pinned host -> device copy of x, W, g and device -> host read of y, dx, dW "
               "every step; copies of neighbouring steps overlap the compute on two copy "
               "streams (two device buffer sets)")
        serial = time_e2e(wl, max(3, min(args.steps, 10)), flush, stream)
        serial_ms = max_over_ranks(sum(serial) / len(serial), world)
    else:
        e2e = time_e2e(wl, max(3, min(args.steps, 10)), flush, stream)
        e2e_ms = serial_ms = max_over_ranks(sum(e2e) / len(e2e), world)
        how = "pinned host copies in and out every step, one stream"
    line["e2e"] = {"value": round(wl.flops * world / (e2e_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": wl.h2d, "d2h_bytes_per_step": wl.d2h,
                   "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps, "how": how,
                   "serial_ms_per_step": round(serial_ms, 4)}
    if not args.no_extras and rank == 0:
        line["rows"] = run_extras(dev, flush, stream, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_rows)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    """The CPU oracle on the same workload: each step is a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = Float8Linear.__new__(Float8Linear)
    wl.T, wl.din, wl.dout = 8192, 2048, 2048
    x, w, g = workloads.float8_linear()
    wl.host_in = [x, w, g]
    wl.name = Float8Linear.name
    # calibrate: size each step's sample so that the whole run takes ~2 min
    _, dt_cal, _ = wl.oracle_sample(256)
    per_row = dt_cal / 256
    rows = int(min(8192, max(64, 120.0 / max(args.steps, 1) / per_row)) // 64 * 64)
    flops_total, secs, sample = 0.0, 0.0, ""
    for _ in range(args.steps):
        f, dt, sample = wl.oracle_sample(rows)
        flops_total += f
        secs += dt
    value = flops_total / secs / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {
        "impl": "reference",
        "metric": "FP8 scaled-GEMM TFLOP/s incl. quantize, % of FP8 peak; quantize GB/s % HBM",
        "value": value, "unit": "TFLOP/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle over fp8 codes)", "data": "synthetic",
        "config": {"workload": wl.name, "tokens": 8192, "d_in": 2048, "d_out": 2048,
                   "scaling": "per-tensor current"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- other workloads --

def time_launches(fns, iters, flush, stream, warmup=3):
    """Mean device ms of each launch in pass order (L2 flushed at the start of
    every pass, a memory-free spin kernel before every launch so the host is
    ahead of the GPU), and their sum as the time of one pass."""
    for _ in range(warmup):
        for _, fn in fns:
            fn()
    torch.cuda.synchronize()
    rec = {}
    for _ in range(iters):
        flush.zero_()
        for label, fn in fns:
            torch.cuda._sleep(SPIN_CYCLES)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            rec.setdefault(label, []).append((s, e))
    torch.cuda.synchronize()
    per = {k: sum(s.elapsed_time(e) for s, e in v) / len(v) for k, v in rec.items()}
    count = {}
    for label, _ in fns:
        count[label] = count.get(label, 0) + 1
    per = {k: v for k, v in per.items()}
    step = sum(per[k] * count[k] for k in per)
    return per, step


def snr_db_dev(x, xhat):
    d = (x.double() - xhat.double())
    return float(10.0 * torch.log10((x.double() ** 2).sum() / (d * d).sum()))


class GroupGemm:
    """Fine-grained FP8 inference GEMM: activations quantized per token in
    1x128 groups (timed), weights in 128x128 blocks (offline), K 7168, N 2048."""

    _w_cache = {}

    def __init__(self, dev, m, sfmt_name, k=7168, n=2048):
        import fp8_quantized_gemm_gb300 as F
        self.name = "group_%s_m%d" % (sfmt_name, m)
        self.m, self.k, self.n = m, k, n
        sfmt = F.SCALE_F32 if sfmt_name == "f32" else F.SCALE_UE8M0
        sdt = torch.float32 if sfmt == F.SCALE_F32 else torch.uint8
        key = (sfmt_name, k, n, str(dev))
        if key not in GroupGemm._w_cache:
            _, w = workloads.fine_grained(1, k=k, n=n)
            wd = w.to(dev)
            wq = torch.empty((n, k), dtype=torch.uint8, device=dev)
            ws = torch.empty(((n + 127) // 128, k // 128), dtype=sdt, device=dev)
            F.fp8_quantize_block(wd, F.E4M3, sfmt, wq, ws)  # offline weight quantization
            GroupGemm._w_cache[key] = (wq, ws)
        self.wq, self.ws = GroupGemm._w_cache[key]
        act, _ = workloads.fine_grained(m, k=k, n=8)
        self.ad = act.to(dev)
        self.aq = torch.empty((m, k), dtype=torch.uint8, device=dev)
        self.asc = torch.empty((k // 128, m), dtype=sdt, device=dev)
        self.y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        self.sfmt, self.F = sfmt, F

    def launches(self):
        F = self.F
        return [("quantize", lambda: F.fp8_quantize_token_group(self.ad, F.E4M3, self.sfmt, self.aq,
                                                                self.asc)),
                ("gemm", lambda: F.fp8_gemm_group(self.aq, self.asc, self.wq, self.ws, self.sfmt,
                                                  self.y))]

    def report(self, per, step, fp8_peak, hbm):
        m, k, n = self.m, self.k, self.n
        flops = 2.0 * m * n * k
        gb = n * k + m * k + m * n * 2 + self.ws.numel() * self.ws.element_size() + \
            self.asc.numel() * self.asc.element_size()
        return {"tflops_incl_quantize": round(flops / (step / 1e3) / 1e12, 2),
                "gemm_tflops": round(flops / (per["gemm"] / 1e3) / 1e12, 2),
                "gemm_frac_fp8_peak": round(flops / (per["gemm"] / 1e3) / 1e12 / fp8_peak, 4),
                "gemm_gbs": round(gb / (per["gemm"] / 1e3) / 1e9, 1),
                "gemm_frac_hbm": round(gb / (per["gemm"] / 1e3) / 1e9 / hbm, 4),
                "quantize_gbs": round((m * k * 3 + self.asc.numel() * self.asc.element_size())
                                      / (per["quantize"] / 1e3) / 1e9, 1),
                "ms": {kk: round(v, 4) for kk, v in per.items()}}


class MoeExperts:
    """Mixture-of-experts layer, 8 experts, 4096 routed tokens (uneven
    counts), N 2048, K 7168: token-group quantization of the activations
    (timed), expert weights in 128x128 blocks (offline), one expert-grouped
    GEMM launch over all experts."""

    def __init__(self, dev, sfmt_name, experts=8, tokens=4096, k=7168, n=2048):
        import fp8_quantized_gemm_gb300 as F
        self.name = "moe_experts_%s_e%d_t%d" % (sfmt_name, experts, tokens)
        self.e, self.t, self.k, self.n = experts, tokens, k, n
        sfmt = F.SCALE_F32 if sfmt_name == "f32" else F.SCALE_UE8M0
        sdt = torch.float32 if sfmt == F.SCALE_F32 else torch.uint8
        act, w, counts = workloads.moe_experts(experts, tokens, n, k)
        self.counts = counts.tolist()
        offsets = torch.cat([torch.zeros(1, dtype=torch.int64), counts.cumsum(0)]).to(torch.int32)
        self.offsets = offsets.to(dev)
        wd = w.to(dev)
        self.wq = torch.empty((experts, n, k), dtype=torch.uint8, device=dev)
        self.ws = torch.empty((experts, (n + 127) // 128, k // 128), dtype=sdt, device=dev)
        for e in range(experts):  # offline weight quantization
            F.fp8_quantize_block(wd[e], F.E4M3, sfmt, self.wq[e], self.ws[e])
        del wd
        self.ad = act.to(dev)
        self.aq = torch.empty((tokens, k), dtype=torch.uint8, device=dev)
        self.asc = torch.empty((k // 128, tokens), dtype=sdt, device=dev)
        self.y = torch.empty((tokens, n), dtype=torch.bfloat16, device=dev)
        self.sfmt, self.F = sfmt, F

    def launches(self):
        F = self.F
        return [("quantize", lambda: F.fp8_quantize_token_group(self.ad, F.E4M3, self.sfmt, self.aq,
                                                                self.asc)),
                ("gemm", lambda: F.fp8_gemm_group_experts(self.aq, self.asc, self.wq, self.ws,
                                                          self.sfmt, self.offsets, self.y))]

    def report(self, per, step, fp8_peak, hbm):
        t, k, n, e = self.t, self.k, self.n, self.e
        flops = 2.0 * t * n * k
        gb = e * n * k + t * k + t * n * 2 + self.ws.numel() * self.ws.element_size() + \
            self.asc.numel() * self.asc.element_size()
        return {"tflops_incl_quantize": round(flops / (step / 1e3) / 1e12, 2),
                "gemm_tflops": round(flops / (per["gemm"] / 1e3) / 1e12, 2),
                "gemm_frac_fp8_peak": round(flops / (per["gemm"] / 1e3) / 1e12 / fp8_peak, 4),
                "gemm_gbs": round(gb / (per["gemm"] / 1e3) / 1e9, 1),
                "tokens_per_expert": self.counts,
                "ms": {kk: round(v, 4) for kk, v in per.items()}}


class TwoLevel:
    """MOSS two-level microscaling GEMM, M = N = K = 8192: amax and two-level
    quantization of both operands, then the block-scaled GEMM."""

    name = "two_level_8192"

    def __init__(self, dev, m=8192, n=8192, k=8192):
        import fp8_quantized_gemm_gb300 as F
        self.F, self.m, self.n, self.k = F, m, n, k
        a, b = workloads.two_level(m=m, n=n, k=k)
        self.ad, self.bd = a.to(dev), b.to(dev)
        self.bufs = []
        for t, r in ((self.ad, m), (self.bd, n)):
            self.bufs.append((t, torch.empty(1, device=dev), torch.empty(1, device=dev),
                              torch.empty((r, k), dtype=torch.uint8, device=dev),
                              F.mx_local_words(r, k, dev)))
        self.y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)

    def launches(self):
        F, out = self.F, []
        for t, am, gl, q, lw in self.bufs:
            out.append(("amax", lambda t=t, am=am: F.fp8_amax(t, am)))
            out.append(("quantize", lambda t=t, am=am, gl=gl, q=q, lw=lw:
                        F.fp8_quantize_mx(t, F.E4M3, am, gl, q, lw)))
        A, B = self.bufs
        out.append(("gemm", lambda: F.fp8_gemm_mx(A[3], A[4], A[2], B[3], B[4], B[2], self.y)))
        return out

    def report(self, per, step, fp8_peak, hbm):
        M, N, K = self.m, self.n, self.k
        flops = 2.0 * M * N * K
        row = {"tflops_incl_quantize": round(flops / (step / 1e3) / 1e12, 2),
               "gemm_tflops": round(flops / (per["gemm"] / 1e3) / 1e12, 2),
               "gemm_frac_fp8_peak": round(flops / (per["gemm"] / 1e3) / 1e12 / fp8_peak, 4),
               "quantize_gbs": round(M * K * (3 + 1 / 32) / (per["quantize"] / 1e3) / 1e9, 1),
               "amax_gbs": round(M * K * 2 / (per["amax"] / 1e3) / 1e9, 1),
               "ms": {kk: round(v, 4) for kk, v in per.items()}}
        row["snr_db"] = self.snr()
        return row

    def snr(self):
        """SNR of A under the three granularities, from the kernels' codes."""
        F, M, K = self.F, self.m, self.k
        dev = self.ad.device
        e4 = torch.float8_e4m3fn
        x = self.ad.float()
        t, am, gl, q, lw = self.bufs[0]
        F.fp8_amax(t, am)
        F.fp8_quantize_mx(t, F.E4M3, am, gl, q, lw)
        loc = lw.view(torch.uint8).view(K // 128, -1, 4)  # [G, Rpad, 4] bytes in word order
        rows_ = torch.arange(M, device=dev)
        pos = (rows_ & ~127) + 4 * (rows_ % 32) + (rows_ % 128) // 32
        r = loc[:, pos, :].permute(1, 0, 2).reshape(M, K // 32).float()
        deq2 = q.view(e4).float().view(M, K // 32, 32) * (gl * torch.exp2(r - 127.0))[:, :, None]
        qt = torch.empty((M, K), dtype=torch.uint8, device=dev)
        st = torch.empty(1, device=dev)
        F.fp8_quantize_tensor(self.ad, F.E4M3, qt, amax_in=am, scale_out=st)
        qg = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sg = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
        F.fp8_quantize_token_group(self.ad, F.E4M3, F.SCALE_F32, qg, sg)
        deqg = qg.view(e4).float().view(M, K // 128, 128) * sg.t()[:, :, None]
        return {"per_tensor": round(snr_db_dev(x, qt.view(e4).float() * st), 3),
                "per_group_1x128": round(snr_db_dev(x, deqg.view(M, K)), 3),
                "two_level": round(snr_db_dev(x, deq2.view(M, K)), 3)}


def extra_workloads(dev):
    for sname in ("f32", "ue8m0"):
        for m in (1, 128, 4096):
            yield GroupGemm(dev, m, sname)
    yield TwoLevel(dev)
    for sname in ("ue8m0", "f32"):
        yield MoeExperts(dev, sname)


def run_swiglu_row(dev, stream, fp8_peak, flush, weight_scaling="delayed"):
    """FP8 SwiGLU MLP training, d 4096, ffn 14336, 16384 tokens, 16 steps
    (inputs drawn on the device from seeded generators); activations and
    gradients with delayed scaling, weights delayed or automatic (MOSS eq. 10)."""
    from fp8_quantized_gemm_gb300.mlp import SwiGLUTrainer
    x, w1, w3, w2 = workloads.swiglu(device=dev)
    tr = SwiGLUTrainer(w1, w3, w2, tokens=x.shape[0], weight_scaling=weight_scaling)
    del w1, w3, w2
    dys = [workloads.swiglu_grad(t, device=dev) for t in range(17)]
    tr.step(x, dys[0])  # warm-up step (kernel attributes, split-K scratch)
    torch.cuda.synchronize()
    steps16 = 16
    fb_ms, opt_ms = [], []
    s0 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for t in range(steps16):
        e1, e2, e3 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e1.record(stream)
        tr.forward_backward(x, dys[t + 1])
        e2.record(stream)
        tr.optimizer_and_state()
        e3.record(stream)
        fb_ms.append((e1, e2))
        opt_ms.append((e2, e3))
    s1 = torch.cuda.Event(enable_timing=True)
    s1.record(stream)
    torch.cuda.synchronize()
    total = s0.elapsed_time(s1)
    fb = sum(a.elapsed_time(b) for a, b in fb_ms) / steps16
    op = sum(a.elapsed_time(b) for a, b in opt_ms) / steps16
    row = {"tflops_incl_quantize": round(tr.flops_per_step * steps16 / (total / 1e3) / 1e12, 2),
           "frac_fp8_peak": round(tr.flops_per_step * steps16 / (total / 1e3) / 1e12 / fp8_peak, 4),
           "ms_per_step": round(total / steps16, 3),
           "ms_forward_backward": round(fb, 3), "ms_adamw_and_state": round(op, 3),
           "tflop_per_step": round(tr.flops_per_step / 1e12, 3),
           "launch": "eager, one API call per kernel"}
    if weight_scaling == "auto":
        # per-tensor cost of the two ways of scaling a weight (MOSS Table 1:
        # just-in-time 0.08-0.54 ms per tensor, automatic 0.02 ms)
        import fp8_quantized_gemm_gb300 as F
        jit, auto = [], []
        for w in tr.w_bf:
            per, _ = time_launches([("jit", lambda w=w: F.fp8_amax(w, tr.w_amax0[0:1]))], 10,
                                   flush, stream)
            jit.append(per["jit"])
            per, _ = time_launches([("auto", lambda: F.fp8_auto_weight_scale(
                tr.w_amax0[0:1], 7, 1e-4, F.E4M3, tr.scale[1:2]))], 10, flush, stream)
            auto.append(per["auto"])
        row["weight_scale_us_per_tensor"] = {
            "jit_amax": round(1e3 * sum(jit) / 3, 2), "automatic": round(1e3 * sum(auto) / 3, 2),
            "weight_bytes": int(tr.w_bf[0].numel() * 2),
            "note": "jit = fp8_amax max-reduction of the bf16 weight after an L2 flush; "
                    "automatic = fp8_auto_weight_scale"}
    del tr, x, dys
    torch.cuda.empty_cache()
    return row


def run_extras(dev, flush, stream, peaks, iters=10):
    import fp8_quantized_gemm_gb300 as F
    fp8_peak, hbm = 2.0 * peaks["bf16_tflops"], peaks["hbm_gbs"]
    out = {}
    for wl in extra_workloads(dev):
        per, step = time_launches(wl.launches(), iters, flush, stream)
        out[wl.name] = wl.report(per, step, fp8_peak, hbm)
        del wl
    out["swiglu_training_delayed_16steps"] = run_swiglu_row(dev, stream, fp8_peak, flush)
    out["swiglu_training_auto_weight_scaling_16steps"] = run_swiglu_row(dev, stream, fp8_peak,
                                                                        flush, "auto")
    hist = torch.zeros(1024, device=dev)
    sc = torch.ones(1, device=dev)
    cur = torch.full((1,), 3.0, device=dev)
    per, _ = time_launches([("update", lambda: F.fp8_delayed_state_update(hist, sc, cur, F.E4M3))],
                           iters, flush, stream)
    out["delayed_state_update_L1024"] = {"us": round(per["update"] * 1e3, 2)}
    return out


PROFILE_WORKLOADS = {
    "float8_linear": lambda dev: Float8Linear(dev),
    "two_level_8192": lambda dev: TwoLevel(dev),
    **{"group_%s_m%d" % (s_, m): (lambda dev, s_=s_, m=m: GroupGemm(dev, m, s_))
       for s_ in ("f32", "ue8m0") for m in (1, 128, 4096)},
    **{"moe_%s" % s_: (lambda dev, s_=s_: MoeExperts(dev, s_)) for s_ in ("f32", "ue8m0")},
}


def run_profile(args):
    """A workload's launch sequence only (warmup + steps passes, no flush
    buffer, no baselines): the command ncu captures use."""
    import fp8_quantized_gemm_gb300 as F
    dev, _, _ = setup_dist()
    wl = PROFILE_WORKLOADS[args.profile](dev)
    for _ in range(args.warmup + args.steps):
        for _, fn in wl.launches():
            fn()
    torch.cuda.synchronize()
    rc, where = F.fp8_get_last_device_error()
    if rc != 0:
        raise RuntimeError("device error %d (where %d)" % (rc, where))
    print("profile run %s: %d passes of %d launches" % (args.profile, args.warmup + args.steps,
                                                        len(wl.launches())))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager launches, not a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=8192)
    ap.add_argument("--profile", default=None, choices=sorted(PROFILE_WORKLOADS),
                    help="run one workload's launch sequence only (for ncu captures); "
                         "prints no bench line")
    args = ap.parse_args()
    if args.profile is not None:
        run_profile(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
