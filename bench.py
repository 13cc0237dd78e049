#!/usr/bin/env python
"""Throughput benchmark of the 8-bit quantized linear (libqlin, C ABI).

A step is one pass over a workload's linears with inputs resident in HBM.  The
default workload is the FP8-E4M3 W8A16 decode sweep on 7B-class shapes
(q_proj 3584->3584, gate_up_proj 3584->37888, down_proj 18944->3584, each at
M in {1, 8, 32, 128, 256}); the metric is quantized-linear GB/s of algorithmic
bytes (8-bit weights + fp32 scales + BF16 activations in + BF16 outputs out).
Two copies of the weights (2 x 217 MB, each larger than the 129 MB L2)
alternate between steps, so every step streams its weights from HBM.

Other workloads (--workload): small, w8a8-3b, prefill, stack-decode,
stack-prefill; prefill-shaped ones report TFLOP/s instead of GB/s.

--impl reference times the CPU oracle (the plain fp64 restatement of the layer)
on a bounded sample of the same workload on the host cores.

Under torchrun (--gpus N > 1) every rank runs an independent replica (the layer
has no exchange step); value is the sum over ranks of units / max elapsed.
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_quantized_linear_gb300 import synth  # noqa: E402

L2_BYTES = 129 * 2 ** 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- workloads
def workload_calls(name: str):
    """List of synth.Linear describing one step of the workload."""
    if name == "decode7b":
        return synth.workload(synth.DECODE7B).linears, synth.DECODE7B
    if name == "small":
        return synth.workload(synth.SMALL).linears, synth.SMALL
    if name == "w8a8-3b":
        return synth.workload(synth.W8A8_3B).linears, synth.W8A8_3B
    if name == "prefill":
        return synth.workload(synth.PREFILL).linears, synth.PREFILL
    if name == "w8a8-dyn-3b":
        return synth.workload(synth.W8A8_DYN_3B).linears, synth.W8A8_DYN_3B
    if name == "stack-decode":
        return synth.stack_linears("decode"), synth.STACK + "-decode"
    if name == "stack-prefill":
        return synth.stack_linears("prefill"), synth.STACK + "-prefill"
    raise SystemExit(f"unknown workload {name}")


def alg_bytes(l) -> int:
    b = l.N * l.K + 4 * l.N + 2 * l.M * l.K + 2 * l.M * l.N
    if l.bias:
        b += 2 * l.N
    return b


def alg_flops(l) -> int:
    return 2 * l.M * l.N * l.K


def is_prefill(name: str) -> bool:
    return name in ("prefill", "stack-prefill")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3][1:5]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[2] for r in rows)}


# ----------------------------------------------------------- GPU workload
class GpuWorkload:
    """Quantized weights, inputs and pre-marshalled C-ABI arguments of one step."""

    def __init__(self, name, dev, copies=2):
        import torch
        from bit_quantized_linear_gb300 import capi
        self.torch, self.capi = torch, capi
        self.lins, self.wl = workload_calls(name)
        self.name = name
        self.dev = dev
        L = capi.lib()
        self.stream = torch.cuda.current_stream()
        sp = ctypes.c_void_p(self.stream.cuda_stream)
        # weights: one quantized copy per distinct (layer, name, K, N, qtype), then `copies` sets
        wkeys = {}
        for l in self.lins:
            wkeys.setdefault((l.workload, l.layer, l.name, l.K, l.N, l.qtype), l)
        self.weight_bytes = sum(l.N * l.K for l in wkeys.values())
        self.copies = copies if self.weight_bytes < 4 * L2_BYTES else 1
        self.wsets = [dict() for _ in range(self.copies)]
        self.scales = {}
        # the 36-layer stack draws its tensors with a seeded device generator
        # (same distributions; host generation of 2.8 G weights would take minutes)
        self.device_gen = name.startswith("stack")
        for key, l in wkeys.items():
            if self.device_gen:
                g = torch.Generator(device=dev)
                g.manual_seed(synth.sub_seed(l.workload, l.layer, f"{l.name}.K{l.K}.N{l.N}", "weight") % (2 ** 63))
                w = torch.randn((l.N, l.K), generator=g, device=dev, dtype=torch.float32) * (1.0 / l.K ** 0.5)
            else:
                w = torch.from_numpy(synth.make_inputs(l, want=("w",))["w"]).to(dev)
            qw, s = capi.quantize_weight(l.qtype, w)
            del w
            self.scales[key] = s
            self.wsets[0][key] = qw
            for c in range(1, self.copies):
                self.wsets[c][key] = qw.clone()
        # activations, calibration scales, bias, outputs
        self.x, self.y, self.bias, self.sx, self.ws = [], [], [], [], []
        self.x_host, self.y_host = [], []
        cache, shared = {}, {}
        def dev_normal(shape, role, l):
            g = torch.Generator(device=dev)
            g.manual_seed(synth.sub_seed(l.workload, l.layer, f"{l.name}.K{l.K}.M{l.M}", role) % (2 ** 63))
            return torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)

        for l in self.lins:
            k = (l.workload, l.layer, l.name, l.K, l.M)
            if self.device_gen:
                t = {"x_dev": dev_normal((l.M, l.K), "act", l)}
                if l.form == "w8a8":
                    t["cal_dev"] = dev_normal((synth.CALIB_ROWS, l.K), "calib", l)
            else:
                if k not in cache:
                    cache[k] = synth.make_inputs(l, want=("x", "cal", "bias"))
                t = cache[k]
            shape_key = (l.form, l.qtype, l.M, l.K, l.N)
            if self.device_gen:
                # the stack's 216 calls are sequential on one stream: outputs, scratch and
                # pinned host staging are shared per shape (each layer keeps its own x)
                xt = t["x_dev"]
                if ("xh",) + shape_key not in shared:
                    shared[("xh",) + shape_key] = xt.cpu().pin_memory()
                    shared[("y",) + shape_key] = torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev)
                    shared[("yh",) + shape_key] = torch.empty((l.M, l.N), dtype=torch.bfloat16).pin_memory()
                self.x_host.append(shared[("xh",) + shape_key])
                self.y.append(shared[("y",) + shape_key])
                self.y_host.append(shared[("yh",) + shape_key])
            else:
                xt = torch.from_numpy(t["x"].view(np.int16)).to(dev).view(torch.bfloat16)
                self.x_host.append(torch.from_numpy(t["x"].view(np.int16)).view(torch.bfloat16).pin_memory())
                self.y.append(torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev))
                self.y_host.append(torch.empty((l.M, l.N), dtype=torch.bfloat16).pin_memory())
            self.x.append(xt)
            self.bias.append(torch.from_numpy(t["bias"].view(np.int16)).to(dev).view(torch.bfloat16)
                             if "bias" in t else None)
            if l.form == "w8a8dyn":
                self.sx.append(None)
                op = capi.QLIN_OP_W8A8_DYNAMIC_LINEAR
            elif l.form == "w8a8":
                cal = t["cal_dev"] if self.device_gen else \
                    torch.from_numpy(t["cal"].view(np.int16)).to(dev).view(torch.bfloat16)
                self.sx.append(capi.act_scale_from_calib(l.qtype, cal))
                del cal
                op = capi.QLIN_OP_W8A8_LINEAR
            else:
                self.sx.append(None)
                op = capi.QLIN_OP_W8A16_LINEAR
            if ("ws",) + shape_key not in shared or not self.device_gen:
                shared[("ws",) + shape_key] = capi.workspace(op, l.qtype, l.M, l.K, l.N, device=dev)
            self.ws.append(shared[("ws",) + shape_key])
            if len(cache) > 8:
                cache.clear()
        torch.cuda.synchronize()
        P = ctypes.c_void_p

        def ptr(t):
            return None if t is None else P(t.data_ptr())

        # pre-marshalled argument tuples: args[copy][i]
        self.fns, self.args = [], [[] for _ in range(self.copies)]
        for i, l in enumerate(self.lins):
            key = (l.workload, l.layer, l.name, l.K, l.N, l.qtype)
            qt = capi.QTYPES[l.qtype]
            ws = self.ws[i]
            wsp, wsb = (None, 0) if ws is None else (ptr(ws), ws.numel())
            if l.form == "w8a8dyn":
                self.fns.append(L.qlin_w8a8_dynamic_linear)
                for c in range(self.copies):
                    self.args[c].append((qt, l.M, l.K, l.N, ptr(self.x[i]), ptr(self.wsets[c][key]),
                                         ptr(self.scales[key]), ptr(self.bias[i]), ptr(self.y[i]), wsp, wsb, sp))
            elif l.form == "w8a16":
                self.fns.append(L.qlin_w8a16_linear)
                for c in range(self.copies):
                    self.args[c].append((qt, l.M, l.K, l.N, ptr(self.x[i]), ptr(self.wsets[c][key]),
                                         ptr(self.scales[key]), ptr(self.bias[i]), ptr(self.y[i]), wsp, wsb, sp))
            else:
                self.fns.append(L.qlin_w8a8_linear)
                for c in range(self.copies):
                    self.args[c].append((qt, l.M, l.K, l.N, ptr(self.x[i]), ptr(self.sx[i]),
                                         ptr(self.wsets[c][key]), ptr(self.scales[key]), ptr(self.bias[i]),
                                         ptr(self.y[i]), wsp, wsb, sp))
        op = {"w8a16": capi.QLIN_OP_W8A16_LINEAR, "w8a8": capi.QLIN_OP_W8A8_LINEAR,
              "w8a8dyn": capi.QLIN_OP_W8A8_DYNAMIC_LINEAR}
        self.kernel = [capi.qlin_kernel_name(op[l.form], l.qtype, l.M, l.K, l.N) for l in self.lins]

    def _capture(self, copy, events=None, e2e=False):
        """CUDA graph of one step on weight copy `copy` (PDL edges between the
        kernels); with `events`, each call is bracketed by external event nodes;
        with `e2e`, host->device copies of the activations and device->host
        copies of the outputs are part of the graph."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            if e2e:
                for i in range(len(self.lins)):
                    self.x[i].copy_(self.x_host[i], non_blocking=True)
            args = self.args[copy]
            for i, fn in enumerate(self.fns):
                if events is not None:
                    events[i][0].record(self.stream)
                st = fn(*args[i])
                if events is not None:
                    events[i][1].record(self.stream)
                if st != 0:
                    raise RuntimeError(f"{self.kernel[i]}: status {self.capi.status_string(st)}")
            if e2e:
                for i in range(len(self.lins)):
                    self.y_host[i].copy_(self.y[i], non_blocking=True)
        return g

    def build_graphs(self, with_events):
        torch = self.torch
        # capture on a side stream; the pre-marshalled stream argument must be the capture stream
        self.stream = torch.cuda.Stream()
        sp = ctypes.c_void_p(self.stream.cuda_stream)
        self.args = [[a[:-1] + (sp,) for a in argset] for argset in self.args]
        torch.cuda.synchronize()
        self.graphs = [self._capture(c) for c in range(self.copies)]
        self.graphs_e2e = [self._capture(c, e2e=True) for c in range(self.copies)]
        self.events = None
        if with_events:
            self.events = [[[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
                            for _ in self.lins] for _ in range(self.copies)]
            self.graphs_ev = [self._capture(c, events=self.events[c]) for c in range(self.copies)]
        torch.cuda.synchronize()

    def run_step(self, step, ev=None):
        args = self.args[step % self.copies]
        for i, fn in enumerate(self.fns):
            if ev is not None:
                ev[i][0].record(self.stream)
            st = fn(*args[i])
            if ev is not None:
                ev[i][1].record(self.stream)
            if st != 0:
                raise RuntimeError(f"{self.kernel[i]}: status {self.capi.status_string(st)}")

    def run_step_e2e(self, step):
        for i in range(len(self.lins)):
            self.x[i].copy_(self.x_host[i], non_blocking=True)
        self.run_step(step)
        for i in range(len(self.lins)):
            self.y_host[i].copy_(self.y[i], non_blocking=True)


def kernel_digest() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "bit_quantized_linear_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, wl: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{wl}:{kernel}")
    if not e or e.get("kernel_digest") != kernel_digest():
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- CPU side
def oracle_sample(name, rows_per_call=1):
    """Bounded oracle sample of one step: every linear of the workload, first
    `rows_per_call` output rows (the oracle still streams the whole weight)."""
    import oracle
    lins, wl = workload_calls(name)
    if name.startswith("stack"):
        lins = lins[:6]  # one layer of the stack
    prepared = []
    for l in lins:
        t = synth.make_inputs(l, want=("w", "cal", "bias"))
        qt = oracle.INT8 if l.qtype == "int8" else oracle.E4M3
        q, s = oracle.quantize_weight(qt, t["w"])
        r = min(l.M, rows_per_call)
        # the first r rows of the workload's activations (the generator draws rows in order)
        x = synth.make_inputs(l, want=("x",), x_rows=r)["x"]
        sx = oracle.act_scale(qt, t["cal"]) if l.form == "w8a8" and "cal" in t else None
        sub = synth.Linear(l.name, l.K, l.N, r, l.qtype, l.form, l.bias, l.outliers, l.workload, l.layer)
        prepared.append((l, sub, qt, q, s, x, sx, t.get("bias")))

    def run():
        for l, sub, qt, q, s, x, sx, b in prepared:
            if l.form == "w8a16":
                oracle.w8a16(qt, x, q, s, b)
            elif l.form == "w8a8dyn":
                qx, sxr = oracle.quantize_act_per_token(qt, x)
                oracle.w8a8_per_token(qt, qx, sxr, q, s, b)
            else:
                qx = oracle.quantize_act(qt, x, sx)
                oracle.w8a8(qt, qx, sx, q, s, b)

    units = sum(alg_flops(p[1]) if is_prefill(name) else alg_bytes(p[1]) for p in prepared)
    desc = (f"{len(prepared)} linears of the workload, first {rows_per_call} output row(s) each "
            f"(the oracle streams every weight once per row)")
    return run, units, desc, oracle.num_threads()


def cpu_baseline(name, unit_scale, unit):
    run, units, desc, cores = oracle_sample(name)
    run()  # warm
    t0 = time.perf_counter()
    n = 0
    while True:
        run()
        n += 1
        if time.perf_counter() - t0 > 10.0 or n >= 20:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": units / dt / unit_scale, "unit": unit, "cores": cores, "kind": "oracle",
            "sample": desc + f"; {n} timed repetitions, {dt:.3f} s each"}


# ------------------------------------------------------- replicas (N > 1)
def max_over_ranks(value: float, device) -> float:
    """Largest `value` over all ranks (the job's wall time is its slowest
    replica's); identity without an initialised process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_step: float, steps: int, world: int, elapsed_max: float, unit_scale: float) -> float:
    """Weak scaling: every replica processes the same per-step units; the job
    processed world x steps x units in the slowest replica's time."""
    return units_per_step * steps * world / elapsed_max / unit_scale


# ------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["qlin", "reference"], default="qlin")
    ap.add_argument("--workload", default="decode7b",
                    choices=["decode7b", "small", "w8a8-3b", "w8a8-dyn-3b", "prefill", "stack-decode",
                             "stack-prefill"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    a = ap.parse_args()
    if a.warmup < 3:
        a.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    prefill = is_prefill(a.workload)
    metric_unit = "TFLOP/s" if prefill else "GB/s"
    metric = ("quantized-linear TOPS (prefill), % of roofline" if prefill
              else "quantized-linear GB/s (decode M<=256), % of roofline")
    lins, wl = workload_calls(a.workload)
    unit_scale = 1e12 if prefill else 1e9

    if a.impl == "reference":
        if rank != 0:
            return
        run, units, desc, cores = oracle_sample(a.workload)
        for _ in range(a.warmup):
            run()
        t0 = time.perf_counter()
        for _ in range(a.steps):
            run()
        dt = (time.perf_counter() - t0) / a.steps
        v = units / dt / unit_scale
        print(json.dumps({
            "impl": "reference", "metric": metric, "value": v, "unit": metric_unit, "n_gpus": 1,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl, "sample": desc},
            "cpu_baseline": {"value": v, "unit": metric_unit, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": metric_unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from bit_quantized_linear_gb300 import capi

    W = GpuWorkload(a.workload, dev)
    n = len(W.lins)
    units_step = sum(alg_flops(l) if prefill else alg_bytes(l) for l in W.lins)
    bytes_step = sum(alg_bytes(l) for l in W.lins)
    flops_step = sum(alg_flops(l) for l in W.lins)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for s in range(a.warmup):
        W.run_step(s)
    torch.cuda.synchronize()
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        ext_events = True
    except TypeError:
        ext_events = False
    W.build_graphs(with_events=ext_events)
    # graph replays launch on torch's current stream: make it the capture stream
    stream_ctx = torch.cuda.stream(W.stream)
    stream_ctx.__enter__()
    for s in range(a.warmup):
        W.graphs[s % W.copies].replay()
    torch.cuda.synchronize()

    # ---- timed region 1: whole steps as CUDA-graph replays (inputs resident) ----
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        t_start.record(W.stream)
        for s in range(a.steps):
            W.graphs[s % W.copies].replay()
        t_end.record(W.stream)
        torch.cuda.synchronize()
        barrier()
    # graph replays do not pass through the host entry points: count the kernels a step launches
    launches = sum(len(k.split("+")) for k in W.kernel) * a.steps
    elapsed = max_over_ranks(t_start.elapsed_time(t_end) / 1e3, dev)
    clocks = clk.summary()
    ms_step = elapsed / a.steps * 1e3
    value = whole_job_value(units_step, a.steps, world, elapsed, unit_scale)

    # ---- timed region 2: per-launch durations (each call bracketed by CUDA events) ----
    dur = np.zeros((a.steps, n))
    if W.events is not None:
        for s in range(a.steps):
            W.graphs_ev[s % W.copies].replay()
            torch.cuda.synchronize()
            evs = W.events[s % W.copies]
            dur[s] = [evs[i][0].elapsed_time(evs[i][1]) / 1e3 for i in range(n)]
        timing = "graph replay with external event nodes around each launch"
    else:
        evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(n)]
               for _ in range(a.steps)]
        torch.cuda.synchronize()
        for s in range(a.steps):
            W.run_step(s, evs[s])
        torch.cuda.synchronize()
        dur = np.array([[evs[s][i][0].elapsed_time(evs[s][i][1]) / 1e3 for i in range(n)] for s in range(a.steps)])
        timing = "stream events around each launch"
    mean_call = dur.mean(axis=0)
    per_kernel = {}
    for i, l in enumerate(W.lins):
        k = W.kernel[i]
        d = per_kernel.setdefault(k, {"time": 0.0, "bytes": 0, "flops": 0, "calls": 0})
        d["time"] += mean_call[i]
        d["bytes"] += alg_bytes(l)
        d["flops"] += alg_flops(l)
        d["calls"] += 1
    dom = max(per_kernel, key=lambda k: per_kernel[k]["time"])
    peaks, peaks_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    bf16 = peaks["bf16_tflops"]
    d = per_kernel[dom]
    if prefill:
        # FP8 operands: measured BF16 peak x the nominal FP8/BF16 ratio (4.5 / 2.25)
        peak = bf16 * 2.0 if W.lins[0].qtype == "e4m3" else bf16
        roof = {"bound": "tensor", "achieved": d["flops"] / d["time"] / 1e12, "peak": peak, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": d["bytes"] / d["time"] / 1e9, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    tr = traffic_for(dom.split("+")[-1], wl)
    roof["traffic"] = tr
    roof["kernel"] = dom
    roof["peak_source"] = f"{peaks_src} (MEASURED_PEAKS.json)" if peaks_src == "measured" else "fallback"
    roof["timing"] = timing
    # roofline time over the whole step: sum_i max(bytes_i / BW, flops_i / peak_i) / measured
    rt = 0.0
    for l in W.lins:
        tpk = (bf16 * 2.0 if (l.form == "w8a8" and l.qtype == "e4m3") else bf16) * 1e12
        rt += max(alg_bytes(l) / (hbm * 1e9), alg_flops(l) / tpk)
    roof["step_roofline_time_frac"] = rt / (mean_call.sum())
    calls = []
    for i, l in enumerate(W.lins):
        calls.append({"name": l.name, "M": l.M, "K": l.K, "N": l.N, "kernel": W.kernel[i],
                      "us": round(mean_call[i] * 1e6, 2),
                      "GB/s": round(alg_bytes(l) / mean_call[i] / 1e9, 1),
                      "TFLOP/s": round(alg_flops(l) / mean_call[i] / 1e12, 1)})

    # ---- end-to-end through the C ABI with host buffers ----
    e2e = None
    if not a.no_e2e:
        for s in range(a.warmup):
            W.graphs_e2e[s % W.copies].replay()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(W.stream)
        for s in range(a.steps):
            W.graphs_e2e[s % W.copies].replay()
        e1.record(W.stream)
        torch.cuda.synchronize()
        et = max_over_ranks(e0.elapsed_time(e1) / 1e3, dev)
        e2e = {"value": whole_job_value(units_step, a.steps, world, et, unit_scale), "unit": metric_unit,
               "h2d_bytes_per_step": int(sum(2 * l.M * l.K for l in W.lins)),
               "d2h_bytes_per_step": int(sum(2 * l.M * l.N for l in W.lins)),
               "how": "CUDA-graph replay: pinned-host activations copied in, the linears, outputs copied out"}

    stream_ctx.__exit__(None, None, None)
    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_baseline(a.workload, unit_scale, metric_unit)

    if rank == 0:
        out = {
            "metric": metric, "value": value, "unit": metric_unit, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("e4m3" if W.lins[0].qtype == "e4m3" else "int8") + ("xbf16" if W.lins[0].form == "w8a16" else "")
                     + "->f32acc->bf16",
            "data": "synthetic",
            "config": {"workload": wl, "linears": n, "bytes_per_step": bytes_step, "flops_per_step": flops_step,
                       "weight_bytes": W.weight_bytes, "weight_copies": W.copies,
                       "l2": (f"{W.copies} alternating weight copies of {W.weight_bytes / 1e6:.0f} MB each "
                              f"(L2 is {L2_BYTES / 2**20:.0f} MiB)"),
                       "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                       "timing": "CUDA-graph replay of whole steps, CUDA events around the K steps"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": int(launches),
            "clocks": clocks,
            "calls": calls,
        }
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
