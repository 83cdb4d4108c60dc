"""Benchmark of the scaled-FP8 GEMM path on GB300.

Default workload (one "step"): the Float8 linear forward + backward with
per-tensor current scaling -- x[8192,2048] (E4M3), W[2048,2048] (E4M3),
grad_out[8192,2048] (E5M2), bf16 in and out: three amax passes, three fused
quantize passes (each also writing the transposed copy the backward GEMMs
read), and the three GEMMs y = x W^T, dx = g W, dW = g^T x.

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
        out_dir = os.path.join(ROOT, "gpurun_out")
        os.makedirs(out_dir, exist_ok=True)
        self.path = os.path.join(out_dir, "clocks_%d.csv" % os.getpid())
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
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

    GEMM operands are K-contiguous ([rows, K]): y = x W^T reads x_q and W_q;
    dx = g W reads g_q and W_q^T; dW = g^T x reads g_q^T and x_q^T.  The
    quantize passes write both layouts in one pass."""

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
        self.xq, self.xqt = torch.empty((T, di), **u8), torch.empty((di, T), **u8)
        self.wq, self.wqt = torch.empty((do, di), **u8), torch.empty((di, do), **u8)
        self.gq, self.gqt = torch.empty((T, do), **u8), torch.empty((do, T), **u8)
        self.amax = torch.empty(3, device=dev)
        self.scale = torch.empty(3, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.y, self.dx, self.dw = torch.empty((T, do), **bf), torch.empty((T, di), **bf), \
            torch.empty((do, di), **bf)
        self.outputs = [self.y, self.dx, self.dw]
        self.host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in self.outputs]
        self.flops = 3 * 2.0 * T * di * do
        n_x, n_w, n_g = T * di, do * di, T * do
        self.n_elems = n_x + n_w + n_g
        # algorithmic bytes per launch: amax reads 2 B/elem; quantize reads
        # 2 B and writes 1 B + 1 B (transposed copy) per element
        self.bytes = {"amax": 2.0 * self.n_elems / 3, "quantize": 4.0 * self.n_elems / 3}
        self.h2d = sum(t.numel() * t.element_size() for t in self.host_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.outputs)

    def launches(self):
        F = self.F
        a, s = self.amax, self.scale
        T, di, do = self.T, self.din, self.dout
        return [
            ("amax", lambda: F.fp8_amax(self.x, a[0:1])),
            ("amax", lambda: F.fp8_amax(self.w, a[1:2])),
            ("amax", lambda: F.fp8_amax(self.g, a[2:3])),
            ("quantize", lambda: F.fp8_quantize_tensor(self.x, F.E4M3, self.xq, amax_in=a[0:1],
                                                       scale_out=s[0:1], q_t=self.xqt)),
            ("quantize", lambda: F.fp8_quantize_tensor(self.w, F.E4M3, self.wq, amax_in=a[1:2],
                                                       scale_out=s[1:2], q_t=self.wqt)),
            ("quantize", lambda: F.fp8_quantize_tensor(self.g, F.E5M2, self.gq, amax_in=a[2:3],
                                                       scale_out=s[2:3], q_t=self.gqt)),
            ("gemm", lambda: F.fp8_gemm_tensor(self.xq, F.E4M3, self.wq, F.E4M3, s[0:1], s[1:2],
                                               self.y)),
            ("gemm", lambda: F.fp8_gemm_tensor(self.gq, F.E5M2, self.wqt, F.E4M3, s[2:3], s[1:2],
                                               self.dx)),
            ("gemm", lambda: F.fp8_gemm_tensor(self.gqt, F.E5M2, self.xqt, F.E4M3, s[2:3], s[0:1],
                                               self.dw)),
        ]

    def upload(self, stream):
        for h, d in zip(self.host_in, (self.x, self.w, self.g)):
            d.copy_(h, non_blocking=True)

    def download(self, stream):
        for d, h in zip(self.outputs, self.host_out):
            h.copy_(d, non_blocking=True)

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
