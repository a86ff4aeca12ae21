"""Benchmark of the MicroQonv quantize-once convolution hot path on B300.

A step is one pass of the whole path over one batch of synthetic input: every
tensor quantized once into 8x8 channel-batch-first blocks, then the forward,
data-gradient and weight-gradient implicit-im2col GEMMs on the packed blocks.

Default workload: the chained 4-layer stack (N=256, 56x56, C 128->128, 3x3,
stride 1, pad 1, bf16 inputs, NVFP4): quantize X0 and W0..W3, forward through
the four layers with the fused epilogue requantizing Y_l into X_{l+1} (its
T_scale from the previous step's amax, Hindsight-style), quantize dY3, then
wgrad + dgrad of layers 3..0, the dgrad epilogue requantizing dX_l straight
into dY_{l-1} the same way (layer 0 writes fp32 dX).

value = algorithmic conv TFLOP/s of the whole step (quantization included in
the step time); per-op throughputs, the quantizer's GB/s and the roofline of
the dominant kernel are reported beside it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                       [--workload NAME]
Multi-GPU (torchrun): every rank runs the same workload on its own GPU
(replicas; no data-path collective), value sums all ranks' work over the
slowest rank's time.
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

import synthetic as S  # noqa: E402

METRIC = "conv fwd/dgrad/wgrad TFLOP/s + quantizer GB/s, % of roofline, 1 B300"
BITS = {"e2m1": 4.125, "e2m3": 6.125, "e4m3": 8.125}
WORKLOADS = {
    "stack4-nvfp4": 4, "stack4-fp6": 5, "resnet32-cifar": 1, "resnet18-224": 2, "yolov8n-640-fp8": 3,
    "tiny-3x3": 0,
}


def packed_bytes(fmt, elems):
    return elems * BITS[fmt] / 8.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of this GPU's clocks and throttle reasons every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        import torch
        self.proc = None
        self.lines = []
        try:
            prop = torch.cuda.get_device_properties(device_index)
            bus = f"{prop.pci_domain_id:08X}:{prop.pci_bus_id:02X}:{prop.pci_device_id:02X}.0"
            self.cmd = ["nvidia-smi", f"--id={bus}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                        "-lms", "200"]
        except Exception:
            self.cmd = None

    def start(self):
        if not self.cmd:
            return
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- timing
class NullTimer:
    def begin(self, name, layer=None):
        pass

    def end(self):
        pass


class OpTimer:
    """CUDA events around each op group, on the current (launching) stream;
    `layer` optionally tags the op with a layer index."""

    def __init__(self):
        import torch
        self.torch = torch
        self.pairs = []
        self.cur = None

    def begin(self, name, layer=None):
        # external: inside a CUDA-graph capture the record becomes an event
        # node that fires on every replay
        e = self.torch.cuda.Event(enable_timing=True, external=True)
        e.record()
        self.cur = (name, layer, e)

    def end(self):
        e = self.torch.cuda.Event(enable_timing=True, external=True)
        e.record()
        self.pairs.append((self.cur[0], self.cur[1], self.cur[2], e))

    def times(self):
        out = {}
        for name, _, a, b in self.pairs:
            out.setdefault(name, []).append(a.elapsed_time(b))
        return out

    def layer_times(self):
        out = {}
        for name, layer, a, b in self.pairs:
            if layer is not None:
                out.setdefault((layer, name), []).append(a.elapsed_time(b))
        return out


# --------------------------------------------------------------- workloads
class StackStep:
    """The chained-stack training step (see module docstring).  wdec: the
    packed weights carry the decoded fp16 copy (written by the quantizer), so
    fwd and dgrad copy the weight operand instead of decoding it per tile."""

    def __init__(self, wl, device, wdec=True):
        import torch
        import microscaling_quantized_convolution_only_b300 as mq
        self.mq, self.torch, self.wl, self.dev = mq, torch, wl, device
        L = wl.layers[0]
        self.L = L
        fmt = wl.fmt
        self.fmt = fmt
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        nl = len(wl.layers)
        # inputs resident in HBM: X0, W0..W3 (bf16), dY3 (bf16)
        self.h_x0 = torch.from_numpy(S.draw_x(wl, 0)).to(tdt)
        self.h_w = [torch.from_numpy(S.draw_w(wl, l)).to(tdt) for l in range(nl)]
        self.h_dy = torch.from_numpy(S.draw_dy(wl, nl - 1)).to(tdt)
        self.x0 = self.h_x0.to(device)
        self.w = [t.to(device) for t in self.h_w]
        self.dy = self.h_dy.to(device)
        self.xq = [mq.Packed(fmt, "act", L.x_shape(), device=device) for _ in range(nl)]
        self.wq = [mq.Packed(fmt, "weight", L.w_shape(), device=device, decoded=wdec) for _ in range(nl)]
        self.gq = [mq.Packed(fmt, "grad", L.y_shape(), device=device) for _ in range(nl)]
        self.y_last = torch.empty((L.Ho, L.Wo, L.Cout, L.N), dtype=torch.float32, device=device)
        self.dx = torch.empty((L.H, L.W, L.Cin, L.N), dtype=torch.float32, device=device)
        self.dw = [torch.empty(L.w_shape(), dtype=torch.float32, device=device) for _ in range(nl)]
        self.ws = torch.empty(mq.wgrad_workspace_bytes(L), dtype=torch.uint8, device=device)
        self.amax = torch.zeros(16, dtype=torch.float32, device=device)        # exact-mode amax outputs
        self.y_stat = torch.ones(nl, dtype=torch.float32, device=device)       # hindsight statistics of Y_l
        self.y_amax = torch.zeros(nl, dtype=torch.float32, device=device)
        self.dx_stat = torch.ones(nl, dtype=torch.float32, device=device)      # ... and of dX_l (l > 0)
        self.dx_amax = torch.zeros(nl, dtype=torch.float32, device=device)
        self.nl = nl
        # accounting
        n_el = int(np.prod(L.x_shape()))
        w_el = int(np.prod(L.w_shape()))
        self.flops = {"fwd": nl * L.flops, "dgrad": nl * L.flops, "wgrad": nl * L.flops}
        in_b = 2 if wl.dtype == "bf16" else 4
        # weight operand bytes of one conv launch: the decoded copy (2 bytes an
        # element) or the packed blocks
        wb = 2 * w_el if wdec else packed_bytes(fmt, w_el)
        self.qbytes = {   # algorithmic bytes: one read of the input + the packed output (+ the decoded copy)
            "quant_bf16": 2 * (n_el * in_b + packed_bytes(fmt, n_el)) +
                          nl * (w_el * in_b + packed_bytes(fmt, w_el) + (2 * w_el if wdec else 0)),
        }
        self.conv_bytes = {
            "fwd": (nl - 1) * (2 * packed_bytes(fmt, n_el) + wb) + (packed_bytes(fmt, n_el) + wb + 4 * n_el),
            "dgrad": (nl - 1) * (2 * packed_bytes(fmt, n_el) + wb) + (packed_bytes(fmt, n_el) + wb + 4 * n_el),
            "wgrad": nl * (2 * packed_bytes(fmt, n_el) + 4 * w_el),
        }
        # amax + quantize of X0 and each W (+ the decoded copy of each W), fwd
        # per layer, amax + quantize of dY, wgrad + split-K reduction and dgrad
        # per layer
        self.launches_per_step = (2 + 2 * nl) + (nl if wdec else 0) + nl + 2 + 2 * nl + nl
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in [self.h_x0, self.h_dy] + self.h_w)
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in self.dw)

    def run(self, tm=None):
        """Enqueue one step on the current stream.  tm: optional OpTimer
        bracketing each op with CUDA events."""
        mq, L, nl = self.mq, self.L, self.nl
        tm = tm or NullTimer()
        # quantize X0 and the weights (exact two-pass statistics)
        tm.begin("quant")
        mq.quantize_cbf(self.x0, "nchw", self.xq[0], amax_out=self.amax[0:1])
        for l in range(nl):
            mq.quantize_cbf(self.w[l], "oihw", self.wq[l], amax_out=self.amax[1 + l:2 + l])
        tm.end()
        # forward: fused requantization of Y_l into X_{l+1}
        for l in range(nl):
            tm.begin("fwd", l)
            if l < nl - 1:
                mq.fwd(L, self.xq[l], self.wq[l], None, rq_out=self.xq[l + 1], rq_amax_in=self.y_stat[l:l + 1],
                       rq_amax_out=self.y_amax[l:l + 1])
            else:
                mq.fwd(L, self.xq[l], self.wq[l], self.y_last)
            tm.end()
        # backward
        tm.begin("quant")
        mq.quantize_cbf(self.dy, "nchw", self.gq[nl - 1], amax_out=self.amax[8:9])
        tm.end()
        for l in range(nl - 1, -1, -1):
            tm.begin("wgrad", l)
            mq.wgrad(L, self.gq[l], self.xq[l], self.dw[l], self.ws)
            tm.end()
            tm.begin("dgrad", l)
            if l > 0:   # fused requantization of dX_l into dY_{l-1}
                mq.dgrad(L, self.wq[l], self.gq[l], None, rq_out=self.gq[l - 1], rq_amax_in=self.dx_stat[l:l + 1],
                         rq_amax_out=self.dx_amax[l:l + 1])
            else:
                mq.dgrad(L, self.wq[l], self.gq[l], self.dx)
            tm.end()
        # hindsight: next step's statistics are this step's measured amax
        self.y_stat.copy_(self.y_amax)
        self.dx_stat.copy_(self.dx_amax)

    def upload(self, pinned):
        """e2e: host -> device copies of the step's inputs."""
        self.x0.copy_(pinned["x0"], non_blocking=True)
        self.dy.copy_(pinned["dy"], non_blocking=True)
        for l in range(self.nl):
            self.w[l].copy_(pinned["w"][l], non_blocking=True)

    def download(self, pinned):
        for l in range(self.nl):
            pinned["dw"][l].copy_(self.dw[l], non_blocking=True)

    # double-buffered input staging for the end-to-end loop: the host copy of
    # the next step's inputs runs on a copy stream during this step's compute
    def new_staging(self):
        return {"x0": self.torch.empty_like(self.x0), "dy": self.torch.empty_like(self.dy),
                "w": [self.torch.empty_like(t) for t in self.w]}

    def upload_to(self, stage, pinned):
        stage["x0"].copy_(pinned["x0"], non_blocking=True)
        stage["dy"].copy_(pinned["dy"], non_blocking=True)
        for l in range(self.nl):
            stage["w"][l].copy_(pinned["w"][l], non_blocking=True)

    def consume(self, stage):
        self.x0.copy_(stage["x0"])
        self.dy.copy_(stage["dy"])
        for l in range(self.nl):
            self.w[l].copy_(stage["w"][l])

    def pinned(self):
        return {"x0": self.h_x0.pin_memory(), "dy": self.h_dy.pin_memory(),
                "w": [t.pin_memory() for t in self.h_w], "dw": [t.cpu().pin_memory() for t in self.dw]}


class LayersStep:
    """Per-layer workloads (configs 0-3): every layer's X, W, dY quantized once
    from fp32/bf16 NCHW/OIHW, then fwd, dgrad and wgrad of every layer.  wdec
    as for StackStep."""

    def __init__(self, wl, device, wdec=True):
        import torch
        import microscaling_quantized_convolution_only_b300 as mq
        self.mq, self.torch, self.wl, self.dev = mq, torch, wl, device
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        self.layers = []
        self.flops = {"fwd": 0, "dgrad": 0, "wgrad": 0}
        self.conv_bytes = {"fwd": 0.0, "dgrad": 0.0, "wgrad": 0.0}
        self.qbytes = {"quant": 0.0}
        self.h2d_bytes = self.d2h_bytes = 0
        in_b = 2 if wl.dtype == "bf16" else 4
        fmt = wl.fmt
        for li, L in enumerate(wl.layers):
            h = [torch.from_numpy(a).to(tdt) for a in (S.draw_x(wl, li), S.draw_w(wl, li), S.draw_dy(wl, li))]
            d = dict(L=L, h=h, x=h[0].to(device), w=h[1].to(device), dy=h[2].to(device),
                     xq=mq.Packed(fmt, "act", L.x_shape(), device=device),
                     wq=mq.Packed(fmt, "weight", L.w_shape(), device=device, decoded=wdec),
                     gq=mq.Packed(fmt, "grad", L.y_shape(), device=device),
                     y=torch.empty((L.Ho, L.Wo, L.Cout, L.N), device=device),
                     dx=torch.empty((L.H, L.W, L.Cin, L.N), device=device),
                     dw=torch.empty(L.w_shape(), device=device),
                     ws=torch.empty(max(16, mq.wgrad_workspace_bytes(L)), dtype=torch.uint8, device=device),
                     amax=torch.zeros(4, device=device))
            self.layers.append(d)
            xe, we, ye = (int(np.prod(s)) for s in (L.x_shape(), L.w_shape(), L.y_shape()))
            for k in self.flops:
                self.flops[k] += L.flops
            wb = 2 * we if wdec else packed_bytes(fmt, we)
            self.conv_bytes["fwd"] += packed_bytes(fmt, xe) + wb + 4 * ye
            self.conv_bytes["dgrad"] += wb + packed_bytes(fmt, ye) + 4 * xe
            self.conv_bytes["wgrad"] += packed_bytes(fmt, ye) + packed_bytes(fmt, xe) + 4 * we
            self.qbytes["quant"] += (xe + we + ye) * in_b + packed_bytes(fmt, xe + we + ye) + (2 * we if wdec else 0)
            self.h2d_bytes += (xe + we + ye) * in_b
            self.d2h_bytes += we * 4
        self.launches_per_step = len(self.layers) * (6 + (1 if wdec else 0) + 1 + 1 + 2)

    def run(self, tm=None):
        mq = self.mq
        tm = tm or NullTimer()
        for li, d in enumerate(self.layers):
            L = d["L"]
            tm.begin("quant", li)
            mq.quantize_cbf(d["x"], "nchw", d["xq"], amax_out=d["amax"][0:1])
            mq.quantize_cbf(d["w"], "oihw", d["wq"], amax_out=d["amax"][1:2])
            mq.quantize_cbf(d["dy"], "nchw", d["gq"], amax_out=d["amax"][2:3])
            tm.end()
            tm.begin("fwd", li)
            mq.fwd(L, d["xq"], d["wq"], d["y"])
            tm.end()
            tm.begin("dgrad", li)
            mq.dgrad(L, d["wq"], d["gq"], d["dx"])
            tm.end()
            tm.begin("wgrad", li)
            mq.wgrad(L, d["gq"], d["xq"], d["dw"], d["ws"])
            tm.end()

    def upload(self, pinned):
        for d, p in zip(self.layers, pinned["in"]):
            for dst, src in zip((d["x"], d["w"], d["dy"]), p):
                dst.copy_(src, non_blocking=True)

    def download(self, pinned):
        for d, p in zip(self.layers, pinned["dw"]):
            p.copy_(d["dw"], non_blocking=True)

    def pinned(self):
        return {"in": [[t.pin_memory() for t in d["h"]] for d in self.layers],
                "dw": [d["dw"].cpu().pin_memory() for d in self.layers]}


def workload(args):
    import dataclasses
    wl = S.WORKLOADS[WORKLOADS[args.workload]]
    if args.batch:
        if args.batch % 8:
            raise SystemExit("--batch must be a multiple of 8")
        wl = dataclasses.replace(wl, name=f"{wl.name}-N{args.batch}",
                                 layers=[S.scaled_layer(L, N=args.batch) for L in wl.layers])
    return wl


def make_step(wl, device, wdec=True):
    return StackStep(wl, device, wdec) if wl.chained else LayersStep(wl, device, wdec)


# -------------------------------------------------------------- GPU arm
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, world, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def time_quantizer(mq, torch, src, layout, role, fmt, dims, flush, reps=8):
    """Median CUDA-event time (ms) of quantizing `src` in single-pass mode
    (statistic supplied: the tensor's own amax) and in exact two-pass mode,
    L2 flushed before each rep; returns {mode: ms}.  Each mode is captured
    once as a CUDA graph holding the flush, the start event, the quantizer
    call and the end event, and timed by replaying it: nothing the host does
    (argument marshalling, tensor-map encoding, a late launch) can fall
    between the events, as it can for an eager launch that reaches the GPU
    after the flush has drained."""
    dev = src.device
    p = mq.Packed(fmt, role, dims, device=dev)
    stat = torch.zeros(1, device=dev)
    aout = torch.zeros(1, device=dev)
    mq.quantize_cbf(src, layout, p, amax_out=stat)
    torch.cuda.synchronize()
    out = {}
    for mode in ("single_pass", "two_pass"):
        e0 = torch.cuda.Event(enable_timing=True, external=True)
        e1 = torch.cuda.Event(enable_timing=True, external=True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            flush.zero_()
            e0.record()
            if mode == "single_pass":
                mq.quantize_cbf(src, layout, p, amax_in=stat, amax_out=aout)
            else:
                mq.quantize_cbf(src, layout, p, amax_out=aout)
            e1.record()
        ts = []
        for i in range(reps + 2):
            g.replay()
            torch.cuda.synchronize()
            if i >= 2:
                ts.append(e0.elapsed_time(e1))
        out[mode] = statistics.median(ts)
        del g
    mq.check_device_status()
    return out


def quantizer_entry(ms, in_bytes, fmt, elems, peaks):
    """GB/s and fraction of the HBM copy peak on the one-read byte count
    (input + packed output); the two-pass figure also on its two-read count."""
    one = in_bytes + packed_bytes(fmt, elems)
    d = {"bytes_one_read": one}
    for mode, t in ms.items():
        gbs = one / (t * 1e-3) / 1e9
        d[mode] = {"us": t * 1e3, "gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]}
    d["two_pass"]["frac_hbm_two_reads"] = (one + in_bytes) / (ms["two_pass"] * 1e-3) / 1e9 / peaks["hbm_gbs"]
    return d


def layer_rows(wl, per_layer, peaks, launch_bound_us=5.0):
    """Per layer and op: time, TFLOP/s and fraction of the roofline (burst
    bf16 and the HBM copy); ops whose roofline time is below launch_bound_us
    are labelled launch-bound (their time is launch and pipeline latency)."""
    rows = []
    for li, L in enumerate(wl.layers):
        if (li, "fwd") not in per_layer:
            break
        row = {"layer": L.name()}
        xe, we, ye = (int(np.prod(sh)) for sh in (L.x_shape(), L.w_shape(), L.y_shape()))
        fb = packed_bytes(wl.fmt, 1)
        byts = {"fwd": fb * (xe + we) + 4 * ye, "dgrad": fb * (we + ye) + 4 * xe, "wgrad": fb * (ye + xe) + 4 * we}
        for op in ("fwd", "dgrad", "wgrad"):
            v = per_layer[(li, op)]
            t = sum(v) / len(v)
            t_flop = L.flops / (peaks["bf16_tflops"] * 1e12)
            t_byte = byts[op] / (peaks["hbm_gbs"] * 1e9)
            row[op] = {"ms": t, "tflops": L.flops / (t * 1e-3) / 1e12, "frac_roofline": max(t_flop, t_byte) / (t * 1e-3),
                       "bound": "tensor" if t_flop >= t_byte else "hbm"}
            if max(t_flop, t_byte) * 1e6 < launch_bound_us:
                row[op]["launch_bound"] = True
        rows.append(row)
    return rows


def extra_workload(name, device, peaks, steps, flush, wdec=True):
    """One more workload after the headline: its whole step as a CUDA graph
    (per-op and per-layer CUDA-event times), and the quantizer alone on each
    of its activation and output-gradient tensors of 8 MB or more."""
    import torch
    import microscaling_quantized_convolution_only_b300 as mq
    wl = S.WORKLOADS[WORKLOADS[name]]
    step = make_step(wl, device, wdec)
    for _ in range(3):
        step.run()
    torch.cuda.synchronize()
    # flush, start event, the step (CUDA events around each op group), end
    # event: one graph, so no host work falls between the events
    graph, tm = torch.cuda.CUDAGraph(), OpTimer()
    e0 = torch.cuda.Event(enable_timing=True, external=True)
    e1 = torch.cuda.Event(enable_timing=True, external=True)
    with torch.cuda.graph(graph):
        flush.zero_()
        e0.record()
        step.run(tm)
        e1.record()
    per_op, per_layer, step_ms = {}, {}, []
    for _ in range(steps):
        graph.replay()
        torch.cuda.synchronize()
        step_ms.append(e0.elapsed_time(e1))
        for g, v in tm.times().items():
            per_op.setdefault(g, []).extend(v)
        for k, v in tm.layer_times().items():
            per_layer.setdefault(k, []).extend(v)
    mq.check_device_status()
    ms = statistics.median(step_ms)
    flops = sum(step.flops.values())
    ops = {}
    for op in ("fwd", "dgrad", "wgrad"):
        t = sum(per_op[op]) / steps
        ops[op] = {"ms_per_step": t, "tflops": step.flops[op] / (t * 1e-3) / 1e12}
    quant = {}
    in_b = 2 if wl.dtype == "bf16" else 4
    tensors = []
    if wl.chained:
        L = wl.layers[0]
        tensors = [("X0", step.x0, "act", L.x_shape()), ("dY3", step.dy, "grad", L.y_shape())]
    else:
        for li, d in enumerate(step.layers):
            L = d["L"]
            tensors += [(f"L{li}.X", d["x"], "act", L.x_shape()), (f"L{li}.dY", d["dy"], "grad", L.y_shape())]
    for tname, t, role, dims in tensors:
        if t.numel() * in_b < 8e6:
            continue
        qms = time_quantizer(mq, torch, t, "nchw", role, wl.fmt, dims, flush)
        quant[tname] = quantizer_entry(qms, t.numel() * in_b, wl.fmt, t.numel(), peaks)
    out = {"ms_per_step": ms, "tflops": flops / (ms * 1e-3) / 1e12, "conv_flops_per_step": flops,
           "element_format": wl.fmt, "input_dtype": wl.dtype, "steps": steps, "ops": ops,
           "layers": layer_rows(wl, per_layer, peaks), "quantizer_per_tensor": quant,
           "execution": "one CUDA graph per step, L2 flushed (256 MB write) before each; quantizer timed alone"}
    del graph, step
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch
    import microscaling_quantized_convolution_only_b300 as mq

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    wl = workload(args)
    step = make_step(wl, device, not args.packed_weights)
    peaks = load_peaks()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)   # > 126 MB L2

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    mq.check_device_status()

    # ---- the step as CUDA graphs: a plain one (timed as a whole) and one with
    #      CUDA events around each op group (per-op times without host gaps)
    graph = None
    timed_graph, tm_graph, whole_graph = None, None, None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step.run()
        timed_graph, tm_graph = torch.cuda.CUDAGraph(), OpTimer()
        with torch.cuda.graph(timed_graph):
            step.run(tm_graph)
        # the timed step as one graph: L2 flush, start event, the step, end
        # event (no host work can fall between the events)
        s0g = torch.cuda.Event(enable_timing=True, external=True)
        s1g = torch.cuda.Event(enable_timing=True, external=True)
        whole_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(whole_graph):
            flush.zero_()
            s0g.record()
            step.run()
            s1g.record()
        graph.replay()
        timed_graph.replay()
        whole_graph.replay()
        torch.cuda.synchronize()

    def one_step():
        if graph is not None:
            graph.replay()
        else:
            step.run()

    groups = ["quant", "fwd", "dgrad", "wgrad"]
    per_kernel = {g: [] for g in groups}
    per_layer = {}
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    for _ in range(args.steps):
        flush.zero_()                                   # L2 flush between steps (outside the timing)
        if timed_graph is not None:
            tm = tm_graph
            timed_graph.replay()
        else:
            tm = OpTimer()
            step.run(tm)
        torch.cuda.synchronize()
        for g, v in tm.times().items():
            per_kernel[g].extend(v)
        for k, v in tm.layer_times().items():
            per_layer.setdefault(k, []).extend(v)

    # ---- device-timed steps (inputs resident in HBM)
    step_ms = []
    for _ in range(args.steps):
        if whole_graph is not None:
            whole_graph.replay()
            torch.cuda.synchronize()
            step_ms.append(s0g.elapsed_time(s1g))
            continue
        flush.zero_()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        one_step()
        s1.record()
        torch.cuda.synchronize()
        step_ms.append(s0.elapsed_time(s1))
    clk = clocks.stop()
    barrier(world)
    mq.check_device_status()

    total_ms = sum(step_ms)
    total_ms_max = max_over_ranks(total_ms, world, device)
    flops_step = sum(step.flops.values())
    value = world * flops_step * args.steps / (total_ms_max * 1e-3) / 1e12

    def mean(v):
        return sum(v) / len(v) if v else float("nan")

    ops = {}
    for op in ("fwd", "dgrad", "wgrad"):
        t_ms = mean(per_kernel[op]) * len(per_kernel[op]) / args.steps    # per step
        n_launch = len(per_kernel[op]) / args.steps
        ops[op] = {"ms_per_step": t_ms, "tflops": step.flops[op] / (t_ms * 1e-3) / 1e12,
                   "gbs": step.conv_bytes[op] / (t_ms * 1e-3) / 1e9, "launches_per_step": n_launch,
                   "ms_per_launch": t_ms / n_launch}
    qt = sum(per_kernel["quant"]) / args.steps
    qbytes = sum(step.qbytes.values())
    ops["quantize"] = {"ms_per_step": qt, "gbs": qbytes / (qt * 1e-3) / 1e9,
                       "frac_hbm": qbytes / (qt * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    # Roofline denominators: the burst bf16 peak (a step lasts milliseconds at
    # full clock, far from the seconds-long power-capped loop of the
    # sustained figure, which is kept as a second fraction) and the HBM copy.
    pk_t, pk_ts = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    for op in ("fwd", "dgrad", "wgrad"):
        t_roof = max(step.flops[op] / (pk_t * 1e12), step.conv_bytes[op] / (peaks["hbm_gbs"] * 1e9))
        t_roof_s = max(step.flops[op] / (pk_ts * 1e12), step.conv_bytes[op] / (peaks["hbm_gbs"] * 1e9))
        ops[op]["frac_roofline"] = t_roof / (ops[op]["ms_per_step"] * 1e-3)
        ops[op]["frac_roofline_sustained"] = t_roof_s / (ops[op]["ms_per_step"] * 1e-3)
        ops[op]["bound"] = "tensor" if step.flops[op] / (pk_t * 1e12) >= \
            step.conv_bytes[op] / (peaks["hbm_gbs"] * 1e9) else "hbm"
    dom = max(("fwd", "dgrad", "wgrad"), key=lambda o: ops[o]["ms_per_step"])
    d = ops[dom]
    traffic = captured_traffic(wl.name, f"conv_{dom}", wl.layers[0].N)
    traffic_kind = ("dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture at a smaller batch, "
                    "scaled by the batch; the reads are exact, the writes a lower bound (output lines still "
                    "in L2 when a launch ends are written back later)")
    if d["bound"] == "tensor":
        achieved = step.flops[dom] / d["launches_per_step"] / (d["ms_per_launch"] * 1e-3) / 1e12
        roof = {"kernel": f"conv_{dom}", "bound": "tensor", "achieved": achieved,
                "peak": pk_t, "unit": "TFLOP/s", "frac": achieved / pk_t, "traffic": traffic,
                "traffic_kind": traffic_kind, "frac_sustained": achieved / pk_ts,
                "peak_source": f"{peaks['source']} bf16 dense, burst (the step runs milliseconds at full clock; "
                               f"fp16 MMA runs at the bf16 rate); frac_sustained uses the sustained figure"}
    else:
        achieved = step.conv_bytes[dom] / d["launches_per_step"] / (d["ms_per_launch"] * 1e-3) / 1e9
        roof = {"kernel": f"conv_{dom}", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "traffic_kind": traffic_kind, "peak_source": f"{peaks['source']} HBM copy"}

    layers_out = layer_rows(wl, per_layer, peaks)
    # the quantizer alone on the headline's largest input, single-pass and exact two-pass
    if wl.chained:
        in_b = 2 if wl.dtype == "bf16" else 4
        qms = time_quantizer(mq, torch, step.x0, "nchw", "act", wl.fmt, wl.layers[0].x_shape(), flush)
        ops["quantize_x0"] = quantizer_entry(qms, step.x0.numel() * in_b, wl.fmt, step.x0.numel(), peaks)

    # ---- end to end through the public API with host buffers
    pinned = step.pinned()
    e2e_ms = []
    if hasattr(step, "new_staging"):
        # Training-loop form: every step copies one step's inputs from pinned
        # host memory (the next step's, on a copy stream, into one of two
        # staging sets) while it computes on the inputs staged by the
        # previous one; the first step's inputs are staged before the timed
        # region, so the K timed steps move K steps' worth of host copies.
        cs = torch.cuda.Stream()
        stages = [step.new_staging(), step.new_staging()]
        ready = [torch.cuda.Event(), torch.cuda.Event()]
        free = [torch.cuda.Event(), torch.cuda.Event()]
        with torch.cuda.stream(cs):
            step.upload_to(stages[0], pinned)
            ready[0].record(cs)
        torch.cuda.synchronize()
        n_e2e = max(1, args.steps)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(n_e2e):
            b, nb = i % 2, (i + 1) % 2
            with torch.cuda.stream(cs):
                cs.wait_event(free[nb])
                step.upload_to(stages[nb], pinned)
                ready[nb].record(cs)
            torch.cuda.current_stream().wait_event(ready[b])
            step.consume(stages[b])
            free[b].record()
            step.run()             # the library's public calls, issued from the host every step
            step.download(pinned)
        t1.record()
        torch.cuda.synchronize()
        e2e_ms = [t0.elapsed_time(t1) / n_e2e] * n_e2e
        del stages
    else:
        for _ in range(max(1, args.steps)):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            step.upload(pinned)
            step.run()             # the library's public calls, issued from the host every step
            step.download(pinned)
            t1.record()
            torch.cuda.synchronize()
            e2e_ms.append(t0.elapsed_time(t1))
    e2e_max = max_over_ranks(sum(e2e_ms), world, device)
    e2e_value = world * flops_step * len(e2e_ms) / (e2e_max * 1e-3) / 1e12
    mq.check_device_status()

    result = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": f"{wl.fmt} codes x e4m3 scales -> fp16 MMA, fp32 accumulate",
        "data": "synthetic (seeded splitmix64/Box-Muller draws with the workload's distributions)",
        "config": {"workload": wl.name, "layers": [L.name() for L in wl.layers], "element_format": wl.fmt,
                   "input_dtype": wl.dtype, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed (256 MB write) before every timed step; inputs also exceed L2",
                   "execution": "eager launches" if graph is None else
                                "one CUDA graph per step holding the L2 flush, the start event, the step and the "
                                "end event; per-op times from a copy of the step's graph with CUDA events around "
                                "each op group",
                   "weights": "packed blocks, decoded per tile" if args.packed_weights else
                              "packed blocks + the decoded fp16 copy the quantizer writes beside them; fwd and "
                              "dgrad copy it as their weight operand",
                   "e2e_inputs": "double-buffered: each step copies the next step's inputs from pinned host "
                                 "memory on a copy stream while it computes" if hasattr(step, "new_staging") else
                                 "copied from pinned host memory at the start of each step",
                   "conv_flops_per_step": flops_step},
        "ops": ops,
        "layers": layers_out,
        "roofline": roof,
        "clocks": clk,
        "gpu_launches": step.launches_per_step * args.steps,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": step.h2d_bytes,
                "d2h_bytes_per_step": step.d2h_bytes, "ms_per_step": e2e_max / len(e2e_ms),
                "launch": "eager calls of the public API every step (host-side argument checks, planning "
                          "and tensor-map encoding inside the timed region)"},
    }
    if world == 1 and not args.no_extra_workloads and not args.batch:
        # every other workload after the headline (per-layer fractions, quantizer per tensor)
        del step, pinned
        torch.cuda.empty_cache()
        extras = {}
        for name in ("tiny-3x3", "resnet32-cifar", "resnet18-224", "yolov8n-640-fp8", "stack4-fp6"):
            if WORKLOADS[name] != WORKLOADS[args.workload]:
                extras[S.WORKLOADS[WORKLOADS[name]].name] = extra_workload(name, device, peaks, 3, flush,
                                                                            not args.packed_weights)
        result["workloads"] = extras
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------- CPU oracle arm
def oracle_sample_step(wl, budget_s, state):
    """A bounded sample of the workload on the CPU oracle: quantize a slice of
    each input tensor, then 7-loop fp64 fwd/dgrad/wgrad outputs of the first
    layer, one by one.  Returns (conv FLOPs done, seconds)."""
    import oracle
    L = wl.layers[0]
    if "ops" not in state:
        rng = np.random.default_rng(0)
        # a batch slice of 8 keeps the sample's tensors small; taps see the full spatial extent
        Ls = S.scaled_layer(L, N=8)
        X = S.draw_x(wl, 0)[:8]
        W = S.draw_w(wl, 0)
        dY = S.draw_dy(wl, len(wl.layers) - 1)[:8]
        state["ops"] = (Ls, X, W, dY)
        state["idx_f"] = rng.integers(0, int(np.prod(Ls.y_shape())), 512)
        state["idx_d"] = rng.integers(0, int(np.prod(Ls.x_shape())), 512)
        state["idx_w"] = rng.integers(0, int(np.prod(Ls.w_shape())), 16)
    Ls, X, W, dY = state["ops"]
    t0 = time.perf_counter()
    qx = oracle.quantize(X, wl.fmt, "act", "nchw")
    qw = oracle.quantize(W, wl.fmt, "weight", "oihw")
    qg = oracle.quantize(dY, wl.fmt, "grad", "nchw")
    Xd, Wd, Gd = oracle.dequantize(qx), oracle.dequantize(qw), oracle.dequantize(qg)
    oracle.conv_fwd_at(Xd, Wd, Ls, state["idx_f"])
    oracle.conv_dgrad_at(Wd, Gd, Ls, state["idx_d"])
    oracle.conv_wgrad_at(Gd, Xd, Ls, state["idx_w"])
    dt = time.perf_counter() - t0
    per_out = 2 * Ls.Cin * Ls.k * Ls.k
    flops = (len(state["idx_f"]) + len(state["idx_d"])) * per_out + len(state["idx_w"]) * 2 * Ls.N * Ls.Ho * Ls.Wo
    return flops, dt, {"quantized_elements": X.size + W.size + dY.size}


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# dominant kernel, averaged over its launches in one step, from an ncu
# capture of the same workload at a smaller batch (profiles/, command there),
# scaled by the batch.  The writes of the captured launches are a lower
# bound (output lines still in L2 when a launch ends are not counted).  Valid
# only while the conv kernels' sources (CONV_SOURCES) are the captured ones.
TRAFFIC = {
    # one step's four launches (three with the fused requantization of dX,
    # whose 13 MB packed output is still in L2 when the launch ends, and the
    # plain one of layer 0 writing 45 MB of fp32 dX); bytes per launch
    ("stack4-56x56-c128-nvfp4", "conv_dgrad"): {"bytes_per_launch": 24978752.0, "batch": 64, "sources_sha1": "800ddd799aaf12c3197c5b536c2f9b783181d5c7"},
    ("stack4-56x56-c128-nvfp4", "conv_fwd"): {"bytes_per_launch": 24996160.0, "batch": 64, "sources_sha1": "800ddd799aaf12c3197c5b536c2f9b783181d5c7"},
    # the four launches alike; the small write term (split-K partials,
    # 0.07 MB) does not grow with the batch but is scaled with it
    ("stack4-56x56-c128-nvfp4", "conv_wgrad"): {"bytes_per_launch": 26687360.0, "batch": 64, "sources_sha1": "800ddd799aaf12c3197c5b536c2f9b783181d5c7"},
}


# the sources the conv kernels are built from (device code, the parameter
# structs, the planners and the launch set-up)
CONV_SOURCES = ["api.cu", "common.cuh", "kernels.h", "conv_halo.cuh", "conv_halo.cu", "conv_halo_fwd_a.cu",
                "conv_halo_fwd_b.cu", "conv_halo_dgrad_a.cu", "conv_halo_dgrad_b.cu"]


def kernel_sources_sha1(root=None, names=None):
    """SHA-1 of the library sources (all of csrc/, or the files `names`) and
    mqconv.h, with comments and blank space removed (editing a comment does
    not invalidate a capture, editing code does)."""
    import glob
    import hashlib
    import re
    here = root or os.path.dirname(os.path.abspath(__file__))
    csrc = os.path.join(here, "microscaling_quantized_convolution_only_b300", "csrc")
    files = sorted(os.path.join(csrc, n) for n in names) if names else sorted(glob.glob(os.path.join(csrc, "*")))
    files.append(os.path.join(here, "include", "mqconv.h"))
    h = hashlib.sha1()
    for f in files:
        with open(f, encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = " ".join(text.split())
        h.update(os.path.basename(f).encode())
        h.update(text.encode())
    return h.hexdigest()


def captured_traffic(workload, kernel, batch):
    t = TRAFFIC.get((workload, kernel))
    if t is None or t["sources_sha1"] != kernel_sources_sha1(names=CONV_SOURCES):
        return None
    return t["bytes_per_launch"] * batch / t["batch"]


def cpu_baseline(wl, budget_s=15.0):
    state = {}
    flops = secs = 0.0
    reps = 0
    while secs < budget_s and reps < 1000:
        f, dt, info = oracle_sample_step(wl, budget_s, state)
        flops += f
        secs += dt
        reps += 1
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    Ls = state["ops"][0]
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": (f"{reps} reps of: quantize X[:8], W, dY[:8] of {Ls.name()} ({info['quantized_elements']} "
                       f"elements) + 512 fwd, 512 dgrad and 16 wgrad outputs by the fp64 7-loop oracle"),
            "seconds": secs}


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    wl = S.WORKLOADS[WORKLOADS[args.workload]]
    state = {}
    for _ in range(args.warmup):
        oracle_sample_step(wl, 0, state)
    flops = secs = 0.0
    for _ in range(args.steps):
        f, dt, info = oracle_sample_step(wl, 0, state)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    Ls = state["ops"][0]
    sample = (f"per step: quantize X[:8], W, dY[:8] of {Ls.name()} + 512 fwd, 512 dgrad and 16 wgrad outputs "
              f"by the fp64 7-loop oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"kind": "oracle", "cores": threads, "sample": sample, "value": value},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["mqconv", "reference"], default="mqconv")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="stack4-nvfp4")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of one CUDA graph per step")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="time only the headline workload (the default also times the other workloads after it)")
    ap.add_argument("--packed-weights", action="store_true",
                    help="convolutions decode the packed weight blocks per tile instead of copying the decoded "
                         "fp16 copy that the quantizer writes beside them")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch N (multiple of 8) for small profiling captures; "
                         "the default runs the workload as specified")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl != "reference":
        print("note: warm-up raised to 3 steps", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
