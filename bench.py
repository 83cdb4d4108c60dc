"""Benchmark of the scaled-FP8 GEMM path on one GB300.

Headline workload (one "step"): one training step of the FP8 SwiGLU MLP with
delayed scaling -- d 4096, ffn 14336, 16384 tokens, the largest configuration:
  h = x W1^T, u = x W3^T, a = silu(h) u, y = a W2^T; da = dy W2, dW2 = dy^T a,
  dh, du from da; dx = dh W1 + du W3, dW1 = dh^T x, dW3 = du^T x;
  AdamW on fp32 master weights; nine amax-history updates.
E4M3 activations and weights, E5M2 gradients, every tensor quantized with the
scale its history left (Flax guide 2.3), SwiGLU fused with the quantization
of its outputs.  Nine GEMMs of 2*16384*4096*14336 flop = 17.32 TFLOP per step.
The step is captured as CUDA graphs of the library's API calls (one per
synthetic gradient buffer; the optimizer's step count lives on the device)
and replayed.

Printed: one JSON line -- the headline metric (FP8 scaled-GEMM TFLOP/s
including quantization), the GEMM roofline against the dense FP8 peak, an
end-to-end number through the public API with the step's inputs copied from
pinned host memory every step, the CPU oracle timed on a bounded sample of
the same step, the clocks sampled during the timed region -- and, under
"rows", every other configuration with its own roofline and CPU baseline.
``--impl reference`` times the CPU oracle on the headline workload instead.

Single GPU only: the path runs on one GPU (multi-GPU is out of scope), so
``--gpus`` other than 1 is an error.

Usage: python bench.py [--gpus 1] [--steps K] [--warmup W] [--impl ours|reference]
                       [--no-extras] [--no-cpu-baseline] [--profile NAME]
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
METRIC = "FP8 scaled-GEMM TFLOP/s incl. quantize, % of FP8 peak; quantize GB/s % HBM"


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


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


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
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
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
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------- timing kit --

SPIN_CYCLES = 400_000  # ~0.2 ms at 2 GHz


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
    step = sum(per[k] * count[k] for k in per)
    return per, step


class CallTimer:
    """Device time of every library call a step makes, by wrapping the
    binding's functions: a memory-free spin kernel is queued before each call
    (so the host enqueues it while the GPU spins) and CUDA events on the
    current stream bracket the call.  `per_step` gives the summed ms per
    label per step."""

    def __init__(self, labels):
        import fp8_quantized_gemm_gb300 as F
        self.F = F
        self.labels = labels  # binding function name -> label
        self.recs = []

    def __enter__(self):
        self.orig = {n: getattr(self.F, n) for n in self.labels}
        for n in self.labels:
            setattr(self.F, n, self._wrap(n))
        return self

    def _wrap(self, name):
        fn, label = self.orig[name], self.labels[name]

        def call(*a, **k):
            torch.cuda._sleep(SPIN_CYCLES // 4)
            st = torch.cuda.current_stream()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(st)
            out = fn(*a, **k)
            e.record(st)
            self.recs.append((label, s, e))
            return out
        return call

    def __exit__(self, *exc):
        for n, fn in self.orig.items():
            setattr(self.F, n, fn)

    def per_step(self, steps):
        torch.cuda.synchronize()
        out = {}
        for label, s, e in self.recs:
            out[label] = out.get(label, 0.0) + s.elapsed_time(e)
        return {k: v / steps for k, v in out.items()}


def roofline_entry(bound, achieved, peak, unit, traffic, note):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": note}


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


def cpu_baseline(sample_fn, min_seconds, max_reps=8, unit="TFLOP/s"):
    """The oracle, as it stands, on a bounded sample: repeated until
    `min_seconds` of CPU work; value = work / time in `unit`."""
    work, dt, reps, desc = 0.0, 0.0, 0, ""
    while reps < max_reps and (dt < min_seconds or reps == 0):
        w, d, desc = sample_fn()
        work, dt, reps = work + w, dt + d, reps + 1
    scale = {"TFLOP/s": 1e-12, "GFLOP/s": 1e-9}[unit]
    return {"value": work / dt * scale, "unit": unit, "cores": host_cores(), "kind": "oracle",
            "sample": "%s; %d repetition(s)" % (desc, reps), "seconds": round(dt, 3),
            "repetitions": reps}


def pinned(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().pin_memory()


def fp8_library_probe(dev, n=8192, reps=20):
    """Dense FP8 throughput of the library GEMM (torch._scaled_mm, E4M3,
    per-tensor scales, bf16 out) at n^3: a reference point beside the roofline
    denominator, not part of the path."""
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        e.record()
        torch.cuda.synchronize()
        ms = s.elapsed_time(e) / reps
        return {"tflops": round(2.0 * n ** 3 / (ms / 1e3) / 1e12, 1), "shape": [n, n, n],
                "call": "torch._scaled_mm E4M3 x E4M3 -> bf16, per-tensor scales, burst of %d"
                        % reps}
    except Exception as exc:  # a library build without FP8 support
        return {"tflops": None, "error": str(exc)[:200]}


# ============================================== headline: SwiGLU training ==

class SwiGLUStep:
    """One FP8 SwiGLU training step with delayed scaling (d 4096, ffn 14336,
    16384 tokens): forward, backward, AdamW and the nine history updates."""

    name = "swiglu_training_delayed_d4096_ffn14336_t16384"
    # kernels each step launches: quantize x, dy (2; the weights' codes come
    # from the previous step's AdamW); GEMMs: the gated h|u launch (its
    # epilogue writes a's codes), y, da|dW2, dx|dW1|dW3 and the accumulating
    # dx += du W3 (5); the fused SwiGLU-backward + quantize pass (1); the nine
    # amax-history updates in one launch (1); AdamW with the next step's
    # weight codes (step advance + update: 2).  The amax clears are memsets,
    # not kernels.
    kernels_per_step = 11
    CALL_LABELS = {"fp8_gemm_tensor_grouped": "gemm", "fp8_quantize_tensor": "quantize",
                   "fp8_swiglu_forward_quantize": "swiglu_quantize",
                   "fp8_swiglu_backward_quantize": "swiglu_quantize",
                   "fp8_adamw_multi": "adamw", "fp8_delayed_state_update": "state_update",
                   "fp8_delayed_state_update_multi": "state_update"}

    def __init__(self, dev, n_dy=16, tokens=16384, d=4096, ffn=14336, weight_scaling="delayed"):
        from fp8_quantized_gemm_gb300.mlp import SwiGLUTrainer
        self.dev, self.T, self.d, self.ffn = dev, tokens, d, ffn
        # drawn on the device from the seeded generators (same distributions
        # as the CPU draws of the parity tests)
        self.x, w1, w3, w2 = workloads.swiglu(device=dev, d=d, ffn=ffn, tokens=tokens)
        self.tr = SwiGLUTrainer(w1, w3, w2, tokens=tokens, weight_scaling=weight_scaling)
        del w1, w3, w2
        self.dys = [workloads.swiglu_grad(t, tokens=tokens, d=d, device=dev)
                    for t in range(n_dy)]
        self.flops = self.tr.flops_per_step
        self.graphs = None

    def eager_step(self, i):
        self.tr.step(self.x, self.dys[i % len(self.dys)])

    def capture(self):
        """One CUDA graph per gradient buffer, each the same API calls."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        self.graphs = []
        for j in range(len(self.dys)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                self.tr.step(self.x, self.dys[j])
            self.graphs.append(g)
        torch.cuda.synchronize()

    def replay(self, i):
        self.graphs[i % len(self.graphs)].replay()

    # ---- the CPU oracle on a bounded sample of the step
    def oracle_sample(self, tokens=256, hidden=512):
        """A sub-MLP of the step: the first `tokens` token rows and the first
        `hidden` hidden units (rows of W1 and W3, columns of W2), with the
        full d; every stage of the step in the oracle, in float64: delayed
        scaling quantization of x, W1, W3, W2, a, dy, dh, du, the nine GEMMs,
        SwiGLU, AdamW and the history updates.  Work counted: the nine GEMMs'
        2 * tokens * d * hidden flop each."""
        from oracle import delayed as OD
        from oracle import gemm as OG
        from oracle import training as OT
        x = self.x[:tokens].float().cpu().numpy()
        dy = self.dys[0][:tokens].float().cpu().numpy()
        w1 = self.tr.w_bf[0][:hidden].float().cpu().numpy()
        w3 = self.tr.w_bf[1][:hidden].float().cpu().numpy()
        w2 = self.tr.w_bf[2][:, :hidden].contiguous().float().cpu().numpy()
        t0 = time.perf_counter()
        st = [OD.DelayedState.initial(1024) for _ in range(9)]

        def inq(i, tensor, fmt):
            q, s, st[i] = OD.in_q(tensor, fmt, st[i])
            return OG.dequant_operand(q, fmt, s)

        xd = inq(0, x, "e4m3")
        w1d, w3d, w2d = inq(1, w1, "e4m3"), inq(4, w3, "e4m3"), inq(7, w2, "e4m3")
        h, u = xd @ w1d.T, xd @ w3d.T
        ad = inq(6, OT.swiglu_forward(h, u).astype(np.float32), "e4m3")
        ad @ w2d.T
        dyd = inq(8, dy, "e5m2")
        da = dyd @ w2d
        dw2 = dyd.T @ ad
        dh, du = OT.swiglu_backward(da, h, u)
        dhd, dud = inq(2, dh.astype(np.float32), "e5m2"), inq(5, du.astype(np.float32), "e5m2")
        dhd @ w1d + dud @ w3d
        for w, g in ((w1, dhd.T @ xd), (w3, dud.T @ xd), (w2, dw2)):
            OT.adamw_step(w, g, np.zeros_like(g), np.zeros_like(g), step=1)
        dt = time.perf_counter() - t0
        flops = 9 * 2.0 * tokens * self.d * hidden
        return flops, dt, ("sub-MLP of one step: %d of %d tokens x %d of %d hidden units, full "
                           "d %d (quantize, 9 GEMMs, SwiGLU, AdamW, histories)"
                           % (tokens, self.T, hidden, self.ffn, self.d))

    # ---- end to end through the public API, host buffers every step
    def e2e(self, steps, n_host=4):
        """Each step copies its inputs, the token batch x and the synthetic
        gradient dy, from pinned host memory, runs the training step through
        the library's API calls (a CUDA graph of them per input set, as the
        headline replays them), and reads the step's FP8 statistics (the nine
        amaxes and the nine scales) back to pinned host memory.  Two device
        input sets alternate so that the next step's copies overlap this
        step's compute (a copy stream; the compute stream waits for them)."""
        tr = self.tr
        hx = pinned(self.x.cpu())
        hdy = [pinned(self.dys[j].cpu()) for j in range(n_host)]
        sets = [(torch.empty_like(self.x), torch.empty_like(self.dys[0])) for _ in range(2)]
        out_host = [(torch.empty(9).pin_memory(), torch.empty(9).pin_memory()) for _ in range(2)]
        comp = torch.cuda.current_stream()
        s_in = torch.cuda.Stream()
        done = [None, None]
        for b in range(2):  # warm
            sets[b][0].copy_(hx)
            sets[b][1].copy_(hdy[b])
            tr.step(*sets[b])
        torch.cuda.synchronize()
        # the step's API calls captured once per input set, as the headline
        # replays them (the copies and the read-back stay outside the graphs)
        side = torch.cuda.Stream()
        side.wait_stream(comp)
        graphs = []
        for b in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                tr.step(*sets[b])
            graphs.append(g)
        torch.cuda.synchronize()
        for g in graphs:  # warm replays
            g.replay()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(comp)
        s_in.wait_stream(comp)
        copies = []
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if done[b] is not None:
                    s_in.wait_event(done[b])  # the step that last read set b is finished
                began = torch.cuda.Event(enable_timing=True)
                began.record(s_in)
                sets[b][0].copy_(hx, non_blocking=True)
                sets[b][1].copy_(hdy[i % n_host], non_blocking=True)
                arrived = torch.cuda.Event(enable_timing=True)
                arrived.record(s_in)
                copies.append((began, arrived))
            comp.wait_event(arrived)
            graphs[b].replay()
            out_host[b][0].copy_(tr.amax, non_blocking=True)
            out_host[b][1].copy_(tr.scale, non_blocking=True)
            done[b] = torch.cuda.Event()
            done[b].record(comp)
        end.record(comp)
        torch.cuda.synchronize()
        ms = start.elapsed_time(end) / steps
        # the copies' own duration inside the loop, beside the compute
        self.h2d_copy_loaded_ms = sorted(a.elapsed_time(z) for a, z in copies)[len(copies) // 2]
        h2d = hx.numel() * hx.element_size() + hdy[0].numel() * hdy[0].element_size()
        d2h = 2 * 9 * 4
        # the host link on its own: one step's input copies with nothing else
        # running (the e2e step is link-bound when this takes longer than the
        # device step)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(comp)
        sets[0][0].copy_(hx, non_blocking=True)
        sets[0][1].copy_(hdy[0], non_blocking=True)
        c1.record(comp)
        torch.cuda.synchronize()
        self.h2d_copy_ms = c0.elapsed_time(c1)
        del sets, hx, hdy, graphs
        return ms, h2d, d2h


def run_headline(args, dev, peaks):
    import fp8_quantized_gemm_gb300 as F
    wl = SwiGLUStep(dev)
    stream = torch.cuda.current_stream()
    for i in range(2):  # kernel attributes and per-device set-up, before any capture
        wl.eager_step(i)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        wl.eager_step(i)
    torch.cuda.synchronize()
    # the timed region: K steps of the API calls issued directly (one call
    # per kernel launch; measured about 2% faster than replaying the same
    # calls from CUDA graphs, which follow below)
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for i in range(args.steps):
            wl.eager_step(args.warmup + i)
        e.record(stream)
        torch.cuda.synchronize()
    total_ms = s.elapsed_time(e)
    rc, where = F.fp8_get_last_device_error()
    if rc != 0:
        raise RuntimeError("device error %d (where %d) during the timed region" % (rc, where))
    value = wl.flops * args.steps / (total_ms / 1e3) / 1e12
    # the same K steps replayed from CUDA graphs of the calls
    wl.capture()
    for i in range(args.warmup):
        wl.replay(i)
    torch.cuda.synchronize()
    gs, ge = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gs.record(stream)
    for i in range(args.steps):
        wl.replay(args.warmup + i)
    ge.record(stream)
    torch.cuda.synchronize()
    graph_ms = gs.elapsed_time(ge) / args.steps
    # device time of each call (the roofline's dominant kernel: the GEMMs)
    reps = 3
    with CallTimer(SwiGLUStep.CALL_LABELS) as ct:
        for i in range(reps):
            wl.eager_step(i)
    per = ct.per_step(reps)
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    fp8_peak_sus = 2.0 * peaks["bf16_tflops_sustained"]
    gemm_tflops = wl.flops / (per["gemm"] / 1e3) / 1e12
    src = "MEASURED_PEAKS.json (%s)" % peaks["source"]
    T, d, ffn = wl.T, wl.d, wl.ffn
    # algorithmic HBM bytes of the standalone passes per step
    qbytes = 3.0 * (2 * T * d)                               # x, dy: 2 B in, 1 B out
    sbytes = (3 * 2 + 2 * 1.0) * T * ffn                     # SwiGLU backward: da, h, u -> dh, du codes
    line = {
        "metric": METRIC,
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8 e4m3/e5m2, fp32 accumulate", "data": "synthetic",
        "config": {"workload": wl.name, "tokens": T, "d": d, "ffn": ffn,
                   "scaling": "delayed (amax history 1024), E4M3 forward / E5M2 gradients",
                   "optimizer": "AdamW lr 1e-4 on fp32 masters",
                   "tflop_per_step": round(wl.flops / 1e12, 3),
                   "inputs": "bf16, seeded (workloads.py), drawn on the device; 16 gradient "
                             "buffers cycled",
                   "l2": "not flushed: inputs larger than L2 (about 6 GB read and written per "
                         "step against the 129 MB L2)",
                   "parallelism": "single GPU"},
        "fraction_of_fp8_peak": round(value / fp8_peak, 4),
        "roofline": dict(roofline_entry(
            "tensor", gemm_tflops, fp8_peak, "TFLOP/s", recorded_traffic("gemm_pair_swiglu_step"),
            "dense FP8 = 2 x measured bf16 burst (%s): each GEMM call timed alone" % src),
            kernel="fp8k::gemm_pair_kernel (the 5 GEMM launches of a step; the gated "
                   "h|u launch includes the SwiGLU forward in its epilogue)",
            units="17.32 TFLOP of GEMMs per step over the GEMM launches' summed device time",
            frac_of_sustained_peak=round(gemm_tflops / fp8_peak_sus, 4),
            sustained_peak=round(fp8_peak_sus, 1)),
        "launch": "the step's API calls issued directly, one call per kernel launch",
        "graph": {"value": round(wl.flops / (graph_ms / 1e3) / 1e12, 2),
                  "ms_per_step": round(graph_ms, 4),
                  "how": "the same steps replayed from CUDA graphs of the calls (one per "
                         "gradient buffer)"},
        "kernel_ms_per_step": {k: round(v, 4) for k, v in per.items()},
        "kernel_timing": "every API call of 3 eager steps bracketed by CUDA events on the "
                         "current stream, a memory-free spin kernel queued before each call",
        "passes_gbs": {
            "quantize": round(qbytes / (per["quantize"] / 1e3) / 1e9, 1),
            "swiglu_quantize": round(sbytes / (per["swiglu_quantize"] / 1e3) / 1e9, 1),
            "adamw": round((29.0 if wl.tr.fuse_wq else 30.0) * 3 * ffn * d
                           / (per["adamw"] / 1e3) / 1e9, 1),
            "hbm_peak": peaks["hbm_gbs"],
            "note": "algorithmic bytes of the standalone passes: quantize x, dy (2 B read, "
                    "1 B codes); the SwiGLU backward reads da, h, u and writes the codes of dh "
                    "and du; AdamW 29 B per weight (p, m, v read and written, dW read, the "
                    "next step's FP8 code written; no bf16 copy, which nothing reads when the "
                    "optimizer writes the codes).  The SwiGLU forward runs in "
                    "the gated h|u GEMM's epilogue and is inside 'gemm'"},
        "clocks": clk.summary(),
        "gpu_launches": wl.kernels_per_step * args.steps,
    }
    e2e_steps = max(3, min(args.steps, 20))
    ms, h2d, d2h = wl.e2e(e2e_steps)
    line["e2e"] = {"value": round(wl.flops / (ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "ms_per_step": round(ms, 4), "steps": e2e_steps,
                   "h2d_copy_alone_ms": round(wl.h2d_copy_ms, 4),
                   "h2d_copy_alone_gbs": round(h2d / (wl.h2d_copy_ms / 1e3) / 1e9, 1),
                   "h2d_copy_beside_compute_ms": round(wl.h2d_copy_loaded_ms, 4),
                   "how": "pinned host -> device copy of the token batch x and the gradient dy "
                          "every step on a copy stream (two device input sets alternate, so "
                          "the next step's copies overlap this step's compute); the step's API "
                          "calls replayed from a CUDA graph per input set, as in the headline; "
                          "device -> host read of the step's nine amaxes and scales; "
                          "the host has one NUMA node, the GPU's"}
    return wl, line


# ================================================================== rows ==

class Float8Linear:
    """Float8 linear forward + backward, per-tensor current scaling (x, W, g
    quantized in one launch; y = x W^T, dx = g W, dW = g^T x in one grouped
    launch that reads the codes K-major or MN-major as each GEMM needs: no
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
        # current scaling reads each input once (2 B/elem), writes its codes (1 B/elem)
        self.bytes = {"quantize": 3.0 * self.n_elems}
        s = self.scale
        self.items = [F.quant_item(self.x, F.E4M3, self.xq, s[0:1], self.amax[0:1]),
                      F.quant_item(self.g, F.E5M2, self.gq, s[2:3], self.amax[2:3]),
                      F.quant_item(self.w, F.E4M3, self.wq, s[1:2], self.amax[1:2])]
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
        return [("quantize", lambda: F.fp8_quantize_tensors(self.items, self.sync)),
                ("gemm", lambda: F.fp8_gemm_tensor_grouped(self.problems))]

    def upload(self):
        for h, d in zip(self.host_in, (self.x, self.w, self.g)):
            d.copy_(h, non_blocking=True)

    def download(self):
        for d, h in zip(self.outputs, self.host_out):
            h.copy_(d, non_blocking=True)

    def oracle_sample(self, rows=2048):
        """The oracle on the first `rows` token rows of x and g and the full W:
        current scaling of the three, the three GEMMs."""
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
        return (3 * 2.0 * rows * self.din * self.dout, dt,
                "first %d of %d token rows (x, g), full W; 3 quantizes + 3 GEMMs"
                % (rows, self.T))


def time_graph(fns, steps, flush):
    """`fns` captured once as a CUDA graph and replayed `steps` times, L2
    flushed before each replay; per-replay device ms."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for fn in fns:
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for fn in fns:
            fn()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        graph.replay()
        e.record(stream)
        times.append((s, e))
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in times]


def float8_linear_row(dev, flush, stream, peaks, args):
    wl = Float8Linear(dev)
    steps = 200
    graph_ms = time_graph([fn for _, fn in wl.launches()], steps, flush)
    value = wl.flops / (sum(graph_ms) / steps / 1e3) / 1e12
    reps = 10
    per, _ = time_launches(wl.launches(), reps, flush, stream)
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    gemm_tflops = wl.flops / (per["gemm"] / 1e3) / 1e12
    q_gbs = wl.bytes["quantize"] / (per["quantize"] / 1e3) / 1e9
    src = "MEASURED_PEAKS.json (%s)" % peaks["source"]
    e2e_steps = 20
    launches = wl.launches()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(e2e_steps):
        wl.upload()
        for _, fn in launches:
            fn()
        wl.download()
    e.record(stream)
    torch.cuda.synchronize()
    e2e_ms = s.elapsed_time(e) / e2e_steps
    row = {
        "tflops_incl_quantize": round(value, 2),
        "ms_per_step": round(sum(graph_ms) / steps, 4),
        "config": {"tokens": wl.T, "d_in": wl.din, "d_out": wl.dout,
                   "scaling": "per-tensor current", "l2": "flushed before every step (512 MiB)",
                   "launch": "CUDA graph of the two API calls, 200 replays"},
        "roofline": roofline_entry("tensor", gemm_tflops, fp8_peak, "TFLOP/s",
                                   recorded_traffic("gemm_pair_grouped"),
                                   "dense FP8 = 2 x measured bf16 burst (%s)" % src),
        "quantize_roofline": roofline_entry("hbm", q_gbs, peaks["hbm_gbs"], "GB/s",
                                            recorded_traffic("quantize_multi"),
                                            "measured HBM copy (%s)" % src),
        "kernel_ms": {k: round(v, 4) for k, v in per.items()},
        "e2e": {"value": round(wl.flops / (e2e_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": wl.h2d, "d2h_bytes_per_step": wl.d2h,
                "ms_per_step": round(e2e_ms, 4),
                "how": "pinned host -> device copy of x, W, g and device -> host copy of y, "
                       "dx, dW every step, one stream"},
    }
    if not args.no_cpu_baseline:
        row["cpu_baseline"] = cpu_baseline(lambda: wl.oracle_sample(), args.cpu_seconds)
    return row


class TinyPerTensor:
    """The Flax guide's 16x32 . 32x64 example (2.1/2.2): current scaling of
    both operands, the per-tensor GEMM, fp32 output.  Launch-bound: microseconds."""

    name = "tiny_per_tensor_16x32x64"

    def __init__(self, dev):
        import fp8_quantized_gemm_gb300 as F
        self.F = F
        a, b = workloads.tiny_per_tensor()
        self.a_host, self.bt_host = a, b.t().contiguous()
        self.a, self.bt = a.to(dev), self.bt_host.to(dev)
        u8 = dict(dtype=torch.uint8, device=dev)
        self.qa, self.qb = torch.empty((16, 32), **u8), torch.empty((64, 32), **u8)
        self.am, self.bm, self.sa, self.sb = (torch.empty(1, device=dev) for _ in range(4))
        self.out = torch.empty((16, 64), dtype=torch.float32, device=dev)
        self.sync = torch.zeros(F.QUANT_SYNC_WORDS, dtype=torch.int32, device=dev)

    def launches(self):
        F = self.F
        return [("amax", lambda: F.fp8_amax(self.a, self.am)),
                ("amax", lambda: F.fp8_amax(self.bt, self.bm)),
                ("quantize", lambda: F.fp8_quantize_tensor(self.a, F.E4M3, self.qa,
                                                           amax_in=self.am, scale_out=self.sa)),
                ("quantize", lambda: F.fp8_quantize_tensor(self.bt, F.E4M3, self.qb,
                                                           amax_in=self.bm, scale_out=self.sb)),
                ("gemm", lambda: F.fp8_gemm_tensor(self.qa, F.E4M3, self.qb, F.E4M3, self.sa,
                                                   self.sb, self.out))]

    def launches_fused(self):
        """The same example with both operands' current scaling (amax, scale,
        codes) in one launch."""
        F = self.F
        items = [F.quant_item(self.a, F.E4M3, self.qa, self.sa),
                 F.quant_item(self.bt, F.E4M3, self.qb, self.sb)]
        return [("quantize", lambda: F.fp8_quantize_tensors(items, self.sync)),
                ("gemm", lambda: F.fp8_gemm_tensor(self.qa, F.E4M3, self.qb, F.E4M3, self.sa,
                                                   self.sb, self.out))]

    def oracle_sample(self):
        from oracle import gemm as OG
        from oracle import quantize as OQ
        t0 = time.perf_counter()
        qa, sa = OQ.quantize_tensor(self.a_host.numpy(), "e4m3")
        qb, sb = OQ.quantize_tensor(self.bt_host.numpy(), "e4m3")
        OG.gemm(OG.dequant_operand(qa, "e4m3", sa), OG.dequant_operand(qb, "e4m3", sb))
        return 2.0 * 16 * 32 * 64, time.perf_counter() - t0, "the whole example"


def tiny_row(dev, flush, stream, args):
    wl = TinyPerTensor(dev)
    graph_ms = time_graph([fn for _, fn in wl.launches()], 200, flush)
    per, _ = time_launches(wl.launches(), 20, flush, stream)
    fused_ms = time_graph([fn for _, fn in wl.launches_fused()], 200, flush)
    row = {"us_per_example": round(statistics.median(graph_ms) * 1e3, 2),
           "launch": "CUDA graph of the five API calls (2 amax, 2 quantize, 1 GEMM), median "
                     "of 200 replays after an L2 flush",
           "us_per_example_two_calls": round(statistics.median(fused_ms) * 1e3, 2),
           "two_calls": "CUDA graph of fp8_quantize_tensors (amax, scale and codes of both "
                        "operands in one launch) and the GEMM, median of 200 replays",
           "eager_us_per_call": {k: round(v * 1e3, 2) for k, v in per.items()},
           "flop": 65536}
    if not args.no_cpu_baseline:
        cb = cpu_baseline(wl.oracle_sample, 1.0, max_reps=5000, unit="GFLOP/s")
        cb["us_per_example"] = round(cb["seconds"] / cb["repetitions"] * 1e6, 1)
        row["cpu_baseline"] = cb
    return row


class GroupGemm:
    """Fine-grained FP8 inference GEMM: activations quantized per token in
    1x128 groups (timed), weights in 128x128 blocks (offline), K 7168, N 2048."""

    _w_cache = {}

    def __init__(self, dev, m, sfmt_name, k=7168, n=2048):
        import fp8_quantized_gemm_gb300 as F
        self.name = "group_%s_m%d" % (sfmt_name, m)
        self.sfmt_name = sfmt_name
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
            GroupGemm._w_cache[key] = (wq, ws, w)
        self.wq, self.ws, self.w_host = GroupGemm._w_cache[key]
        act, _ = workloads.fine_grained(m, k=k, n=8)
        self.act_host = act
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

    _w_oracle = {}

    def oracle_sample(self, rows=256):
        """The oracle on the first min(M, rows) activation rows: token-group
        quantization and the per-group GEMM against the offline-quantized
        weights (the weight quantization is not timed, as on the GPU)."""
        from oracle import gemm as OG
        from oracle import quantize as OQ
        r = min(self.m, rows)
        if self.sfmt_name not in GroupGemm._w_oracle:
            qb, sb = OQ.quantize_block(self.w_host.float().numpy(), "e4m3", self.sfmt_name)
            GroupGemm._w_oracle[self.sfmt_name] = OG.dequant_operand(
                qb, "e4m3", OQ.expand(OQ.group_scale_values(sb, self.sfmt_name),
                                      self.n, self.k, 128, 128))
        wdq = GroupGemm._w_oracle[self.sfmt_name]
        act = self.act_host[:r].float().numpy()
        t0 = time.perf_counter()
        qa, sa = OQ.quantize_token_group(act, "e4m3", self.sfmt_name)
        a = OG.dequant_operand(qa, "e4m3", OQ.expand(OQ.group_scale_values(sa, self.sfmt_name),
                                                     r, self.k, 1, 128))
        OG.gemm(a, wdq)
        dt = time.perf_counter() - t0
        return 2.0 * r * self.n * self.k, dt, "%d of %d activation rows" % (r, self.m)

    def graph_timing(self, flush, hbm, copies=14, steps=7):
        """Decode-style timing: one CUDA graph of back-to-back calls, each on
        its own copy of the weights (the copies together exceed L2), replayed
        after an L2 flush; the mean per call of the GEMM alone and of a
        quantize + GEMM pair (consecutive layers of a decode step)."""
        F = self.F
        wqs = [self.wq.clone() for _ in range(copies)]
        wss = [self.ws.clone() for _ in range(copies)]
        gemm = [(lambda i=i: F.fp8_gemm_group(self.aq, self.asc, wqs[i], wss[i], self.sfmt,
                                              self.y)) for i in range(copies)] * 2
        quant = lambda: F.fp8_quantize_token_group(self.ad, F.E4M3, self.sfmt, self.aq, self.asc)
        pairs = []
        for fn in gemm:
            pairs += [quant, fn]
        g_ms = sorted(time_graph(gemm, steps, flush))[steps // 2] / len(gemm)
        p_ms = sorted(time_graph(pairs, steps, flush))[steps // 2] / len(gemm)
        del wqs, wss
        gb = self.gemm_bytes()
        return {"gemm_us": round(g_ms * 1e3, 2), "gemm_gbs": round(gb / (g_ms / 1e3) / 1e9, 1),
                "gemm_frac_hbm": round(gb / (g_ms / 1e3) / 1e9 / hbm, 4),
                "quantize_plus_gemm_us": round(p_ms * 1e3, 2),
                "how": "CUDA graph of %d back-to-back calls over %d weight copies (%.0f MB, "
                       "more than L2), L2 flushed before each replay; median of %d replays, "
                       "per call" % (len(gemm), copies, copies * self.n * self.k / 1e6, steps)}

    def gemm_bytes(self):
        return self.n * self.k + self.m * self.k + self.m * self.n * 2 + \
            self.ws.numel() * self.ws.element_size() + self.asc.numel() * self.asc.element_size()

    def report(self, per, step, fp8_peak, hbm):
        m, k, n = self.m, self.k, self.n
        flops = 2.0 * m * n * k
        gb = self.gemm_bytes()
        return {"tflops_incl_quantize": round(flops / (step / 1e3) / 1e12, 2),
                "gemm_tflops": round(flops / (per["gemm"] / 1e3) / 1e12, 2),
                "gemm_frac_fp8_peak": round(flops / (per["gemm"] / 1e3) / 1e12 / fp8_peak, 4),
                "gemm_gbs": round(gb / (per["gemm"] / 1e3) / 1e9, 1),
                "gemm_frac_hbm": round(gb / (per["gemm"] / 1e3) / 1e9 / hbm, 4),
                "quantize_gbs": round((m * k * 3 + self.asc.numel() * self.asc.element_size())
                                      / (per["quantize"] / 1e3) / 1e9, 1),
                "ms": {kk: round(v, 4) for kk, v in per.items()}}


class GroupGemm32(GroupGemm):
    """The fine-grained GEMM with (32, 32) weight blocks and 1 x 32 activation
    groups, FP32 scales (Transformers fine-grained FP8, 八 and 四): activation
    quantization timed, weights offline, K 7168, N 2048."""

    def __init__(self, dev, m, k=7168, n=2048):
        import fp8_quantized_gemm_gb300 as F
        self.name = "group32_f32_m%d" % m
        self.sfmt_name = "f32"
        self.m, self.k, self.n, self.F = m, k, n, F
        act, w = workloads.fine_grained(m, k=k, n=n)
        self.act_host, self.w_host = act, w
        self.wq = torch.empty((n, k), dtype=torch.uint8, device=dev)
        self.ws = torch.empty(((n + 31) // 32, k // 32), dtype=torch.float32, device=dev)
        F.fp8_quantize_block32_f32(w.to(dev), F.E4M3, self.wq, self.ws)  # offline
        self.ad = act.to(dev)
        self.aq = torch.empty((m, k), dtype=torch.uint8, device=dev)
        self.asc = torch.empty((k // 32, m), dtype=torch.float32, device=dev)
        self.y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)

    def launches(self):
        F = self.F
        return [("quantize", lambda: F.fp8_quantize_token_group32(self.ad, F.E4M3, F.SCALE_F32,
                                                                  self.aq, self.asc)),
                ("gemm", lambda: F.fp8_gemm_group32(self.aq, self.asc, self.wq, self.ws, self.y))]

    def oracle_sample(self, rows=256):
        from oracle import gemm as OG
        from oracle import quantize as OQ
        r = min(self.m, rows)
        if "b32" not in GroupGemm._w_oracle:
            qb, sb = OQ.quantize_block(self.w_host.float().numpy(), "e4m3", "f32", block=32)
            GroupGemm._w_oracle["b32"] = OG.dequant_operand(
                qb, "e4m3", OQ.expand(np.asarray(sb, np.float64), self.n, self.k, 32, 32))
        wdq = GroupGemm._w_oracle["b32"]
        act = self.act_host[:r].float().numpy()
        t0 = time.perf_counter()
        qa, sa = OQ.quantize_token_group(act, "e4m3", "f32", group=32)
        a = OG.dequant_operand(qa, "e4m3", OQ.expand(np.asarray(sa, np.float64), r, self.k, 1, 32))
        OG.gemm(a, wdq)
        dt = time.perf_counter() - t0
        return 2.0 * r * self.n * self.k, dt, "%d of %d activation rows" % (r, self.m)


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
        self.a_host, self.b_host = a, b
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

    def oracle_sample(self, rows=128):
        """The oracle on the first `rows` rows of A and of B: two-level
        quantization of both slices (global factors over the slices) and their
        GEMM."""
        from oracle import gemm as OG
        from oracle import quantize as OQ
        a = self.a_host[:rows].float().numpy()
        b = self.b_host[:rows].float().numpy()
        t0 = time.perf_counter()
        deq = []
        for x in (a, b):
            q, loc, s = OQ.quantize_two_level(x, "e4m3")
            deq.append(OG.dequant_operand(q, "e4m3", OQ.expand(
                OQ.two_level_scale_values(loc, s), rows, self.k, 1, 32)))
        OG.gemm(deq[0], deq[1])
        dt = time.perf_counter() - t0
        return 2.0 * rows * rows * self.k, dt, ("first %d rows of A and of B (K %d): two-level "
                                                "quantization of both, their GEMM" % (rows, self.k))

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

        def snr_db(ref, xhat):
            dd = ref.double() - xhat.double()
            return float(10.0 * torch.log10((ref.double() ** 2).sum() / (dd * dd).sum()))
        return {"per_tensor": round(snr_db(x, qt.view(e4).float() * st), 3),
                "per_group_1x128": round(snr_db(x, deqg.view(M, K)), 3),
                "two_level": round(snr_db(x, deq2.view(M, K)), 3)}


def run_swiglu_auto_row(dev, flush, stream):
    """The training step with MOSS automatic weight scaling (section 5, eq.
    10) for the weights, 16 eager steps; and the per-tensor cost of the two
    ways of scaling a weight (MOSS Table 1: just-in-time 0.08-0.54 ms per
    tensor, automatic 0.02 ms)."""
    import fp8_quantized_gemm_gb300 as F
    wl = SwiGLUStep(dev, n_dy=4, weight_scaling="auto")
    tr = wl.tr
    wl.eager_step(0)
    torch.cuda.synchronize()
    steps16 = 16
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for t in range(steps16):
        wl.eager_step(t + 1)
    s1.record(stream)
    torch.cuda.synchronize()
    total = s0.elapsed_time(s1)
    row = {"tflops_incl_quantize": round(wl.flops * steps16 / (total / 1e3) / 1e12, 2),
           "ms_per_step": round(total / steps16, 3), "launch": "eager, one API call per kernel"}
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
    del wl, tr
    torch.cuda.empty_cache()
    return row


def run_extras(dev, flush, stream, peaks, args):
    import fp8_quantized_gemm_gb300 as F
    fp8_peak, hbm = 2.0 * peaks["bf16_tflops"], peaks["hbm_gbs"]
    out = {}
    out["tiny_per_tensor_16x32x64"] = tiny_row(dev, flush, stream, args)
    out["float8_linear_fwd_bwd"] = float8_linear_row(dev, flush, stream, peaks, args)
    for sname in ("f32", "ue8m0"):
        for m in (1, 128, 4096):
            wl = GroupGemm(dev, m, sname)
            per, step = time_launches(wl.launches(), 10, flush, stream)
            row = wl.report(per, step, fp8_peak, hbm)
            if m <= 128:
                row["graph"] = wl.graph_timing(flush, hbm)
            if not args.no_cpu_baseline:
                row["cpu_baseline"] = cpu_baseline(wl.oracle_sample, args.cpu_seconds / 2)
            out[wl.name] = row
            del wl
    # the decode-sized rows between 1 and 128 (the few-row kernel up to 64)
    few = {}
    for sname in ("f32", "ue8m0"):
        for m in (16, 32, 64):
            wl = GroupGemm(dev, m, sname)
            few["%s_m%d" % (sname, m)] = wl.graph_timing(flush, hbm)
            del wl
    out["group_few_rows_graph"] = few
    for m in (128, 4096):
        wl = GroupGemm32(dev, m)
        per, step = time_launches(wl.launches(), 10, flush, stream)
        row = wl.report(per, step, fp8_peak, hbm)
        if not args.no_cpu_baseline:
            row["cpu_baseline"] = cpu_baseline(wl.oracle_sample, args.cpu_seconds / 2)
        out[wl.name] = row
        del wl
    wl = TwoLevel(dev)
    per, step = time_launches(wl.launches(), 10, flush, stream)
    row = wl.report(per, step, fp8_peak, hbm)
    if not args.no_cpu_baseline:
        row["cpu_baseline"] = cpu_baseline(wl.oracle_sample, args.cpu_seconds)
    out[wl.name] = row
    del wl
    for sname in ("ue8m0", "f32"):
        wl = MoeExperts(dev, sname)
        per, step = time_launches(wl.launches(), 10, flush, stream)
        out[wl.name] = wl.report(per, step, fp8_peak, hbm)
        del wl
    torch.cuda.empty_cache()
    out["swiglu_training_auto_weight_scaling_16steps"] = run_swiglu_auto_row(dev, flush, stream)
    hist = torch.zeros(1024, device=dev)
    sc = torch.ones(1, device=dev)
    cur = torch.full((1,), 3.0, device=dev)
    per, _ = time_launches([("update", lambda: F.fp8_delayed_state_update(hist, sc, cur, F.E4M3))],
                           10, flush, stream)
    out["delayed_state_update_L1024"] = {"us": round(per["update"] * 1e3, 2)}
    return out


# ================================================================== arms ==

def run_ours(args):
    peaks = load_peaks()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    wl, line = run_headline(args, dev, peaks)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(lambda: wl.oracle_sample(), 2 * args.cpu_seconds)
    del wl
    torch.cuda.empty_cache()
    line["roofline"]["library_fp8_probe"] = fp8_library_probe(dev)
    if not args.no_extras:
        stream = torch.cuda.current_stream()
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        line["rows"] = run_extras(dev, flush, stream, peaks, args)
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The CPU oracle on the headline workload: each step a bounded sample of
    the training step (a sub-MLP of the first t tokens and h hidden units),
    sized so that the whole run takes about two minutes."""
    wl = SwiGLUStep.__new__(SwiGLUStep)
    wl.T, wl.d, wl.ffn = 16384, 4096, 14336
    wl.x, w1, w3, w2 = workloads.swiglu()
    wl.dys = [workloads.swiglu_grad(0)]

    class _Weights:  # the weights the sample slices, as the trainer holds them
        w_bf = [w1, w3, w2]
    wl.tr = _Weights()
    _, dt_cal, _ = wl.oracle_sample(tokens=128, hidden=512)
    budget = 100.0 / max(args.steps + args.warmup, 1)
    # the sample's cost grows about linearly with hidden (weights) at fixed tokens
    hidden = int(max(128, min(1024, 512 * budget / max(dt_cal, 1e-3))) // 128 * 128)
    tokens = 128
    for _ in range(args.warmup):
        wl.oracle_sample(tokens=tokens, hidden=hidden)
    flops_total, secs, sample = 0.0, 0.0, ""
    for _ in range(args.steps):
        f, dt, sample = wl.oracle_sample(tokens=tokens, hidden=hidden)
        flops_total += f
        secs += dt
    value = flops_total / secs / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle over fp8 codes)", "data": "synthetic",
        "config": {"workload": SwiGLUStep.name, "tokens": 16384, "d": 4096, "ffn": 14336,
                   "scaling": "delayed (amax history 1024), E4M3 forward / E5M2 gradients"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": host_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PROFILE_WORKLOADS = {
    "float8_linear": lambda dev: Float8Linear(dev),
    "two_level_8192": lambda dev: TwoLevel(dev),
    "tiny": lambda dev: TinyPerTensor(dev),
    **{"group_%s_m%d" % (s_, m): (lambda dev, s_=s_, m=m: GroupGemm(dev, m, s_))
       for s_ in ("f32", "ue8m0") for m in (1, 16, 64, 128, 4096)},
    **{"moe_%s" % s_: (lambda dev, s_=s_: MoeExperts(dev, s_)) for s_ in ("f32", "ue8m0")},
    **{"group32_f32_m%d" % m: (lambda dev, m=m: GroupGemm32(dev, m)) for m in (128, 4096)},
}


def run_profile(args):
    """A workload's launch sequence only (warmup + steps passes, no flush
    buffer, no baselines): the command ncu captures use.  'swiglu' runs eager
    training steps of the headline workload."""
    import fp8_quantized_gemm_gb300 as F
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    if args.profile in ("swiglu", "swiglu_t4096"):
        wl = SwiGLUStep(dev, n_dy=2, tokens=16384 if args.profile == "swiglu" else 4096)
        for i in range(args.warmup + args.steps):
            wl.eager_step(i)
        n = SwiGLUStep.kernels_per_step
    else:
        wl = PROFILE_WORKLOADS[args.profile](dev)
        for _ in range(args.warmup + args.steps):
            for _, fn in wl.launches():
                fn()
        n = len(wl.launches())
    torch.cuda.synchronize()
    rc, where = F.fp8_get_last_device_error()
    if rc != 0:
        raise RuntimeError("device error %d (where %d)" % (rc, where))
    print("profile run %s: %d passes of %d launches" % (args.profile, args.warmup + args.steps, n))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=5.0,
                    help="CPU seconds of oracle work per row baseline (headline: twice this)")
    ap.add_argument("--profile", default=None,
                    choices=sorted(PROFILE_WORKLOADS) + ["swiglu", "swiglu_t4096"],
                    help="run one workload's launch sequence only (for ncu captures); "
                         "prints no bench line")
    args = ap.parse_args()
    if args.gpus != 1:
        sys.stderr.write("bench.py: the scaled-FP8 path runs on one GPU; multi-GPU runs are "
                         "not built (got --gpus %d)\n" % args.gpus)
        sys.exit(2)
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
