#!/usr/bin/env python3
"""Benchmark: NCHW conv2d TFLOP/s (and the broadcast's GB/s) on one GB300.

Headline workload (the default line): the five ResNet-50 bottleneck layers at
N=256, fp16 in / fp32 accumulate / fp16 out, (CI,CO,H,W,K,stride,pad) =
(64,64,56,56,1,1,0), (64,64,56,56,3,1,1), (64,256,56,56,1,1,0),
(512,512,7,7,3,1,1), (256,512,28,28,1,2,0).  One step runs every layer once
through the C ABI; the metric is the step's total FLOP over its device time.
The same run then measures the other workloads and reports each under
"workloads" on the same line: the fused 3x3 conv + exp(conv + bias) (N=32),
the [128,256,32,32] broadcast (with its A/B against the flat schedule and the
general [B0,P,B1] form), the depthwise layers (N=64), the fp32 batch-1 layer
sweep and the N=1 512->512 7x7 layer.  --workload W --only measures one.

Timing: W untimed warm-up steps; K timed steps, each bracketed by CUDA events
on the launch stream, with an L2 flush (a 512 MB write, then a 512 MB read that
drains the write's dirty lines) between steps outside the events.  A second pass of K steps, also timed, adds the library's own
per-kernel event records and an event after every layer; the roofline and the
per-layer figures come from it (those events serialise the launches, so it is
reported separately as profiled_ms_per_step).  `e2e` repeats the
step with host buffers: pinned host->device copies of every layer's inputs and
device->host copies of its output inside the timed region, on two copy streams
that overlap the convs.  Layers and images are independent problems, so each
layer moves in four batch slices (each with its own plan), the layers with the
most output first: the first outputs leave while later inputs still arrive.  `cpu_baseline` times
the CPU oracle on this host on a bounded sample of the same workload.  With
--impl reference the CPU oracle is the measured arm.

Multi-GPU: the layers and images are independent, so N ranks run N replicas of
the step with no exchange (weak scaling); value = all ranks' work / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "conv2d TFLOP/s per shape and % of roofline at 1 GB300; broadcast HBM GB/s"
L2_FLUSH_BYTES = 512 << 20
E2E_CHUNKS = 4        # batch slices per layer in the end-to-end step


# ---------------------------------------------------------------- workloads
def workload_specs(name):
    from broadcast_implicit_gemm_gb300 import synth
    return {
        "sweep_fp32": synth.SWEEP_FP32,
        "resnet_last": synth.RESNET_LAST,
        "resnet50_fp16": synth.RESNET50_FP16,
        "fused": synth.FUSED_CONV,
        "depthwise_fp16": synth.DEPTHWISE_FP16,
    }[name]


def out_hw(s):
    return ((s.H + 2 * s.pad - s.K) // s.stride + 1, (s.W + 2 * s.pad - s.K) // s.stride + 1)


def conv_flops(s):
    Ho, Wo = out_hw(s)
    return 2.0 * s.N * s.CO * Ho * Wo * (s.CI // s.groups) * s.K * s.K


def _touched(n, k, stride, pad, nout):
    return len({o * stride + r - pad for o in range(nout) for r in range(k)
                if 0 <= o * stride + r - pad < n})


def conv_bytes(s):
    """Algorithmic bytes: the input pixels some tap reads, the kernel, the output, once each."""
    Ho, Wo = out_hw(s)
    e_in = 4 if s.in_dtype == "f32" else 2
    e_out = 4 if s.out_dtype == "f32" else 2
    pix = _touched(s.H, s.K, s.stride, s.pad, Ho) * _touched(s.W, s.K, s.stride, s.pad, Wo)
    b = s.N * s.CI * pix * e_in + s.CO * (s.CI // s.groups) * s.K * s.K * e_in
    b += s.N * s.CO * Ho * Wo * e_out
    if s.epi != "none":
        b += 4 * s.CO
    return float(b)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "sm_max_mhz": 2070.0, "source": "fallback"}


def pipe_peak(peaks, in_dtype, kind):
    """TFLOP/s of the pipe a kernel uses.  fp16 = bf16 (measured); tf32 = measured bf16 x
    the nominal dense ratio 1.1/2.25; FP32 FMA = 152 SMs x 128 lanes x 2 x max clock."""
    if kind == "simt":
        return 152 * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12, "fp32 fma (derived)"
    if in_dtype == "f32":
        return peaks["bf16"] * 1.1 / 2.25, f"tf32 (bf16 {peaks['source']} x 1.1/2.25)"
    return peaks["bf16"], f"bf16/fp16 ({peaks['source']})"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = str(gpu_index)
        try:
            import torch
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(gpu_index).uuid)
        except Exception:
            pass
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", prefix="bench_clocks_", suffix=".csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # the first sample lands before the timed region starts
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 3.0 and os.path.getsize(self.f.name) == 0:
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = self.f.read().splitlines()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in rows:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm
class ConvStep:
    """Plans (timed search, cached) and device buffers for every layer of a workload."""

    def __init__(self, specs, device, search=1, seed=0):
        import torch

        import broadcast_implicit_gemm_gb300 as bg
        from broadcast_implicit_gemm_gb300 import synth
        self.bg, self.torch = bg, torch
        self.specs = specs
        self.items = []
        self.marks = None
        # Every layer's inputs (data, kernel, bias) sit back to back, 256-byte
        # aligned, in one pinned host buffer and one device buffer, so that the
        # end-to-end step moves each layer's inputs with a single copy.
        inputs = [synth.conv_inputs(s, seed + i) for i, s in enumerate(specs)]
        def align(n):
            return (n + 255) // 256 * 256
        layout, off = [], 0
        for x, w, b in inputs:
            segs = []
            for t in (x, w, b):
                if t is None:
                    segs.append(None)
                    continue
                nb = t.numel() * t.element_size()
                segs.append((off, nb, t.dtype, tuple(t.shape)))
                off = align(off + nb)
            layout.append(segs)
        self.stage_h = torch.empty(max(off, 256), dtype=torch.uint8).pin_memory()
        self.stage_d = torch.empty(max(off, 256), dtype=torch.uint8, device=device)

        def view(buf, seg):
            o, nb, dt, shape = seg
            return buf[o:o + nb].view(dt).view(shape)

        for i, (s, (x, w, b), segs) in enumerate(zip(specs, inputs, layout)):
            for t, seg in zip((x, w, b), segs):
                if seg is not None:
                    view(self.stage_h, seg).copy_(t)
            Ho, Wo = out_hw(s)
            plan = bg.conv2d_nchw_plan(s.N, s.H, s.W, s.CO, s.CI, s.K, s.K, s.stride, s.pad,
                                       s.groups, bg.DTYPE_CODES[s.in_dtype],
                                       bg.DTYPE_CODES[s.out_dtype], bg.EPI_NAMES[s.epi], search)
            out = torch.empty((s.N, s.CO, Ho, Wo), dtype=synth.TORCH_DTYPES[s.out_dtype],
                              device=device)
            first = segs[0][0]
            last = max(sg[0] + sg[1] for sg in segs if sg is not None)
            item = {
                "spec": s, "plan": plan, "info": plan.describe(),
                "x": view(self.stage_d, segs[0]), "w": view(self.stage_d, segs[1]),
                "b": view(self.stage_d, segs[2]) if segs[2] is not None else None,
                "in_d": self.stage_d[first:last], "in_h": self.stage_h[first:last],
                "out": out, "out_h": torch.empty(out.shape, dtype=out.dtype).pin_memory(),
            }
            # The end-to-end step moves a layer in E2E_CHUNKS batch slices, each
            # with its own plan, so that the first outputs leave while later
            # inputs are still arriving (images are independent problems).
            k = E2E_CHUNKS if s.N % E2E_CHUNKS == 0 and s.N >= E2E_CHUNKS else 1
            nc = s.N // k
            # every slice must start on a 16-byte boundary, as the library requires
            if (segs[0][1] // s.N * nc) % 16 or (out[0].numel() * out.element_size() * nc) % 16:
                k, nc = 1, s.N
            if k > 1:
                cplan = bg.conv2d_nchw_plan(nc, s.H, s.W, s.CO, s.CI, s.K, s.K, s.stride, s.pad,
                                            s.groups, bg.DTYPE_CODES[s.in_dtype],
                                            bg.DTYPE_CODES[s.out_dtype], bg.EPI_NAMES[s.epi],
                                            search)
            else:
                cplan = plan
            xo, xnb = segs[0][0], segs[0][1]
            wb_first = segs[1][0]
            item["e2e"] = {
                "plan": cplan,
                # the kernel and bias, then the data slices, each one copy
                "wb_d": self.stage_d[wb_first:last], "wb_h": self.stage_h[wb_first:last],
                "x_d": [self.stage_d[xo + j * xnb // k: xo + (j + 1) * xnb // k] for j in range(k)],
                "x_h": [self.stage_h[xo + j * xnb // k: xo + (j + 1) * xnb // k] for j in range(k)],
                "x": [item["x"][j * nc:(j + 1) * nc] for j in range(k)],
                "out": [out[j * nc:(j + 1) * nc] for j in range(k)],
                "out_h": [item["out_h"][j * nc:(j + 1) * nc] for j in range(k)],
            }
            self.items.append(item)
        # layers with the most output bytes first: the device-to-host copies,
        # the longer direction, start early and stay busy
        self.e2e_order = sorted(self.items, key=lambda it: -it["out"].numel() * it["out"].element_size())
        self.stage_d.copy_(self.stage_h)
        torch.cuda.synchronize()

    def run(self, stream):
        for i, it in enumerate(self.items):
            self.bg.conv2d_nchw_run(it["plan"], it["x"], it["w"], it["b"], 1e-5, it["out"], stream)
            if self.marks is not None:
                ev = self.torch.cuda.Event(enable_timing=True)
                ev.record(stream)
                self.marks.append((i, ev))

    def run_e2e(self, stream):
        """The step from pinned host buffers: every layer's kernel and bias, then
        its batch slices, go in on a copy-in stream; each slice's conv runs on
        `stream` once it has landed, and its output comes back on a copy-out
        stream, so copies overlap the convs and the two directions overlap each
        other.  The step ends on `stream` when the last output is on the host."""
        torch = self.torch
        if getattr(self, "copy_streams", None) is None:
            self.copy_streams = (torch.cuda.Stream(), torch.cuda.Stream())
        h2d, d2h = self.copy_streams
        h2d.wait_stream(stream)          # the previous step is done with the input buffers
        landed = []
        with torch.cuda.stream(h2d):
            for it in self.e2e_order:
                e = it["e2e"]
                e["wb_d"].copy_(e["wb_h"], non_blocking=True)
                evs = []
                for xd, xh in zip(e["x_d"], e["x_h"]):
                    xd.copy_(xh, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(h2d)
                    evs.append(ev)
                landed.append(evs)
        for it, evs in zip(self.e2e_order, landed):
            e = it["e2e"]
            for j, ev in enumerate(evs):
                stream.wait_event(ev)
                self.bg.conv2d_nchw_run(e["plan"], e["x"][j], it["w"], it["b"], 1e-5, e["out"][j],
                                        stream)
                done = torch.cuda.Event()
                done.record(stream)
                d2h.wait_event(done)
                with torch.cuda.stream(d2h):
                    e["out_h"][j].copy_(e["out"][j], non_blocking=True)
        stream.wait_stream(d2h)

    def h2d_bytes(self):
        # the bytes the end-to-end step copies: each layer's kernel and bias, and its data
        return sum(it["e2e"]["wb_h"].numel() + sum(x.numel() for x in it["e2e"]["x_h"])
                   for it in self.items)

    def d2h_bytes(self):
        return sum(it["out"].numel() * it["out"].element_size() for it in self.items)

    def work(self):
        return sum(conv_flops(it["spec"]) for it in self.items)


class BcastStep:
    def __init__(self, device, seed=0):
        import torch

        import broadcast_implicit_gemm_gb300 as bg
        from broadcast_implicit_gemm_gb300 import synth
        self.bg, self.torch = bg, torch
        self.shape = synth.BCAST_SHAPE
        N, C, H, W = self.shape
        self.var_h = synth.bcast_var(C, seed).pin_memory()
        self.var = self.var_h.to(device)
        self.out = torch.empty(self.shape, dtype=torch.float32, device=device)
        self.out_h = torch.empty(self.shape, dtype=torch.float32).pin_memory()
        self.items = []
        self.marks = None

    def run(self, stream):
        N, C, H, W = self.shape
        self.bg.bcast_nchw_run(N, C, H, W, self.bg.BC_EXP, self.var, 1e-5, self.out, self.bg.F32,
                               stream)

    def run_op(self, stream, op, flat):
        N, C, H, W = self.shape
        fn = self.bg.bcast_nchw_run_flat if flat else self.bg.bcast_nchw_run
        fn(N, C, H, W, op, self.var, 1e-5, self.out, self.bg.F32, stream)

    def run_e2e(self, stream):
        self.var.copy_(self.var_h, non_blocking=True)
        self.run(stream)
        self.out_h.copy_(self.out, non_blocking=True)

    def work(self):
        return float(self.out.numel() * 4 + self.var.numel() * 4)

    def h2d_bytes(self):
        return self.var.numel() * 4

    def d2h_bytes(self):
        return self.out.numel() * 4


def bg_long_rows(B1, esize=4):
    """Whether the library runs [B0,P,B1] on its per-channel kernel (rows of at
    least 1 KB) rather than its short-row kernel."""
    return B1 * esize >= 1024


class L2Flush:
    """Evicts the previous step's data from L2 between timed steps: a write of
    a buffer four times L2's size, then a read of a second one, so that the
    write's dirty lines are written back during the read -- before the next
    step's events, not inside its first layer -- and L2 is left holding clean
    lines of neither the workload's inputs nor its outputs."""

    def __init__(self, torch, device):
        self.wr = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.torch = torch

    def __call__(self):
        self.wr.fill_(1)
        self.torch.sum(self.rd)


def timed_steps(step_fn, steps, torch, stream, flush):
    """Per-step CUDA event pairs (ms), with an L2 flush before each step."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush()
            a.record(stream)
            step_fn(stream)
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs], evs


def sources_sha(names):
    """Digest of the kernel sources a traffic figure was measured on."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "broadcast_implicit_gemm_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if its sources still match."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{kernel}@{workload}")
    except Exception:
        return None
    if not rec:
        return None
    try:
        h = sources_sha(rec["sources"])
    except (OSError, KeyError):
        return None
    return rec["bytes_per_launch"] if h == rec["sources_sha"] else None


def kernel_work(name, it):
    """Algorithmic (flop, bytes) of one layer's launch of kernel `name`, or None."""
    s, info = it["spec"], it["info"]
    e_in = 4 if s.in_dtype == "f32" else 2
    Ho, Wo = out_hw(s)
    if name.startswith("umma_conv"):
        return (conv_flops(s), conv_bytes(s)) if name == "umma_conv_" + info.get("amode", "") else None
    if name.startswith("simt_conv"):
        return (conv_flops(s), conv_bytes(s)) if info["kind"] == "simt" else None
    if name == "pack_operands" and info.get("amode") == "nhwc":
        return (0.0, 2.0 * (s.N * s.CI * s.H * s.W + s.CO * s.CI * s.K * s.K) * e_in)
    if name == "pack_nhwc" and info.get("amode") == "nhwc":
        return (0.0, 2.0 * s.N * s.CI * s.H * s.W * e_in)
    if name == "pack_weights" and info.get("amode") == "nhwc":
        return (0.0, 2.0 * s.CO * s.CI * s.K * s.K * e_in)
    if name == "splitk_reduce" and info.get("split", 1) > 1:
        out = s.N * s.CO * Ho * Wo
        return (0.0, out * 4.0 * info["split"] + out * (4 if s.out_dtype == "f32" else 2))
    return None


def kernel_roofline(name, prof, step, peaks, args, workload):
    """Roofline of kernel `name`: its algorithmic work per launch over its mean launch time."""
    n, tms = prof[name]
    works = [(kernel_work(name, it), it) for it in step.items]
    works = [(w, it) for w, it in works if w is not None]
    flop = sum(w[0] for w, _ in works) * args.steps / n
    byts = sum(w[1] for w, _ in works) * args.steps / n
    per_launch_s = tms / n / 1e3
    kind = "simt" if name.startswith("simt") else "umma"
    in_dt = works[0][1]["spec"].in_dtype if works else "f32"
    tpk, src = pipe_peak(peaks, in_dt, kind)
    t_flop = flop / (tpk * 1e12)
    t_byte = byts / (peaks["hbm"] * 1e9)
    if flop > 0 and t_flop >= t_byte:
        ach = flop / per_launch_s / 1e12
        r = {"bound": "tensor" if kind == "umma" else "alu", "achieved": ach, "peak": tpk,
             "unit": "TFLOP/s", "frac": ach / tpk, "peak_source": src}
    else:
        ach = byts / per_launch_s / 1e9
        r = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s",
             "frac": ach / peaks["hbm"], "peak_source": peaks["source"] + " copy bandwidth"}
    r.update({"kernel": name, "launches": n, "avg_launch_us": per_launch_s * 1e6,
              "flop_per_launch": flop, "bytes_per_launch": byts,
              "roofline_frac": max(t_flop, t_byte) / per_launch_s,
              "traffic": traffic_for(name, workload)})
    return r


def cpu_baseline(workload, specs, budget_s=12.0):
    """The oracle as it stands, on this host's cores, on a bounded sample of the workload."""
    import oracle
    from broadcast_implicit_gemm_gb300 import synth
    lib = oracle.load()
    cores = oracle.num_threads(lib)
    if workload == "bcast":
        N, C, H, W = synth.BCAST_SHAPE
        n_s = 8
        var = synth.bcast_var(C, 0).numpy()
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.bcast_nchw(n_s, C, H, W, oracle.BC_EXP, var, lib=lib)
            reps += 1
            if time.perf_counter() - t0 > budget_s or reps >= 50:
                break
        dt = (time.perf_counter() - t0) / reps
        return {"value": n_s * C * H * W * 4 / dt / 1e9, "unit": "GB/s", "cores": 1,
                "kind": "oracle",
                "sample": f"[{n_s},{C},{H},{W}] of [{N},{C},{H},{W}] (fp32 bytes), {reps} reps"}
    sample = [(s if s.N <= 2 else s.with_batch(1), i) for i, s in enumerate(specs)]
    inputs = [(s, synth.conv_inputs(s, i)) for s, i in sample]
    flops = sum(conv_flops(s) for s, _ in inputs)
    t0 = time.perf_counter()
    reps = 0
    while True:
        for s, (x, w, b) in inputs:
            oracle.conv2d_nchw(x, w, stride=s.stride, pad=s.pad, groups=s.groups, bias=b,
                               epi=oracle.EPI_BIAS_EXP if s.epi == "bias_exp" else oracle.EPI_NONE,
                               nthreads=cores, lib=lib)
        reps += 1
        if time.perf_counter() - t0 > budget_s or reps >= 200:
            break
    dt = (time.perf_counter() - t0) / reps
    names = ", ".join(s.name for s, _ in sample)
    note = ""
    if any(s.N > 2 for s in specs):
        note = (f"; layers of batch {max(s.N for s in specs)} timed at N=1 (the oracle's time "
                f"grows linearly in N, so its TFLOP/s rate is the full batch's)")
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(sample)} layers ({names}); {reps} passes of {dt * 1e3:.1f} ms{note}"}


def reduce_max(value, dist, device):
    """The largest of the ranks' values (each rank's timed total: the job takes
    as long as its slowest replica); the value itself on one rank."""
    if not dist:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(work_per_rank, world, ms_per_step, scale):
    """Whole-job throughput: every rank runs the same step (weak scaling), so
    the job does world x the per-rank work in the slowest rank's time."""
    return work_per_rank * world / (ms_per_step / 1e3) / scale


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as td
        if args.impl == "reference":
            td.init_process_group("gloo")
        else:
            import torch
            torch.cuda.set_device(local)
            td.init_process_group("nccl")
        dist = td
    return world, rank, local, dist


def run_reference(args, world, rank):
    """The CPU oracle as the measured arm (rank 0 only)."""
    if rank != 0:
        return 0
    specs = None if args.workload == "bcast" else workload_specs(args.workload)
    if specs is not None and args.layer:
        specs = [x for x in specs if x.name == args.layer]
    for _ in range(args.warmup):
        cpu_baseline(args.workload, specs, budget_s=0.0)
    budget = max(0.2, min(2.0, 120.0 / max(1, args.steps)))
    per = [cpu_baseline(args.workload, specs, budget_s=budget) for _ in range(args.steps)]
    v = statistics.median(p["value"] for p in per)
    unit = per[0]["unit"]
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload},
        "cpu_baseline": {"value": v, "unit": unit, "cores": per[0]["cores"], "kind": "oracle",
                         "sample": per[0]["sample"]},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def warm(step_fn, n, torch, stream):
    for _ in range(n):
        with torch.cuda.stream(stream):
            step_fn(stream)
    torch.cuda.synchronize()


def measure(name, args, device, stream, flush, peaks, world, dist, local):
    """One workload: plans, warm-up, the timed pass, the profiled pass, the
    end-to-end pass.  Returns the fields of its JSON line."""
    import torch

    import broadcast_implicit_gemm_gb300 as bg
    if name == "bcast":
        step = BcastStep(device)
        unit, scale = "GB/s", 1e9
    else:
        specs = workload_specs(name)
        if args.layer:
            specs = [x for x in specs if x.name == args.layer]
            if not specs:
                raise SystemExit(f"no layer {args.layer} in {name}")
        if args.batch:
            specs = [x.with_batch(args.batch) for x in specs]
        step = ConvStep(specs, device, search=0 if args.no_search else 1)
        unit, scale = "TFLOP/s", 1e12

    warm(step.run, args.warmup, torch, stream)
    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    # timed pass: step events only, so consecutive kernels overlap their
    # launches (programmatic dependent launch) as they would in use
    times, _ = timed_steps(step.run, args.steps, torch, stream, flush)
    # profiled pass over the same steps: the library's per-kernel events and an
    # event after every layer (these serialise the launches)
    bg.bigemm_profile_enable(True)
    step.marks = []
    ptimes, evs = timed_steps(step.run, args.steps, torch, stream, flush)
    marks, step.marks = step.marks, None
    prof = bg.bigemm_profile_read()
    bg.bigemm_profile_enable(False)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    if bg.bigemm_last_device_error() != 0:
        raise SystemExit(f"a device wait timed out during the timed region of {name}")

    total_ms = reduce_max(sum(times), dist, device)   # the slowest rank's time
    ms_per_step = total_ms / args.steps
    value = job_rate(step.work(), world, ms_per_step, scale)

    # end to end through the public call, host buffers in and out
    warm(step.run_e2e, 2, torch, stream)
    e2e_steps = max(3, min(args.steps, 20))
    e2e_times, _ = timed_steps(step.run_e2e, e2e_steps, torch, stream, flush)
    e2e_ms = reduce_max(sum(e2e_times), dist, device) / e2e_steps
    e2e_value = job_rate(step.work(), world, e2e_ms, scale)

    line = {
        "value": value, "unit": unit, "ms_per_step": ms_per_step,
        "gpu_launches": sum(v[0] for v in prof.values()), "clocks": clk,
        "profiled_ms_per_step": sum(ptimes) / args.steps,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": step.h2d_bytes(),
                "d2h_bytes_per_step": step.d2h_bytes(), "ms_per_step": e2e_ms},
    }
    if name == "bcast":
        line["dtype"] = "f32"
        line["config"] = {"workload": "bcast_exp_[128,256,32,32]_fp32", "op": "exp",
                          "l2": "output (134 MB) larger than L2; flushed between steps (512 MB write, 512 MB read)"}
        n, tms = prof.get("bcast_nchw", (args.steps, total_ms))
        ach = step.work() / (tms / n / 1e3) / 1e9
        # A/B: the per-channel mapping against the flat fused-index schedule, per op
        ab = {}
        for opname, op in (("exp", bg.BC_EXP), ("rsqrt", bg.BC_RSQRT), ("recip", bg.BC_RECIP),
                           ("copy", bg.BC_COPY)):
            res = {}
            for flat in (False, True):
                fn = (lambda st, o=op, f=flat: step.run_op(st, o, f))
                warm(fn, 3, torch, stream)
                tt, _ = timed_steps(fn, max(5, min(args.steps, 20)), torch, stream, flush)
                res["flat" if flat else "per_channel"] = step.work() / (sum(tt) / len(tt) / 1e3) / 1e9
            ab[opname] = {"per_channel_gbs": res["per_channel"], "flat_gbs": res["flat"],
                          "speedup": res["per_channel"] / res["flat"]}
        line["bcast_ab"] = ab
        # the general form [1,P,1] => [B0,P,B1] (bcast_run), exp to fp32, on
        # short, single-element and long rows
        gen = []
        for B0, P, B1 in synth_bcast_general():
            gvar = bcast_var_dev(P, device)
            gout = torch.empty((B0, P, B1), dtype=torch.float32, device=device)
            fn = (lambda st, a=(B0, P, B1), v=gvar, o=gout:
                  bg.bcast_run(*a, bg.BC_EXP, v, 1e-5, o, bg.F32, st))
            warm(fn, 3, torch, stream)
            tt, _ = timed_steps(fn, max(5, min(args.steps, 20)), torch, stream, flush)
            gbs = (gout.numel() * 4 + P * 4) / (sum(tt) / len(tt) / 1e3) / 1e9
            gen.append({"shape": [B0, P, B1], "gbs": gbs, "frac": gbs / peaks["hbm"],
                        "kernel": "bcast_nchw" if bg_long_rows(B1) else "bcast_rows"})
            del gout
        line["bcast_general"] = gen
        line["roofline"] = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s",
                            "frac": ach / peaks["hbm"], "kernel": "bcast_nchw", "launches": n,
                            "avg_launch_us": tms / n * 1e3,
                            "peak_source": peaks["source"] + " copy bandwidth",
                            "traffic": traffic_for("bcast_nchw", name)}
    else:
        kinds = sorted({it["info"]["kind"] for it in step.items})
        in_dt = step.items[0]["spec"].in_dtype
        line["dtype"] = "tf32" if in_dt == "f32" and kinds == ["umma"] else in_dt
        line["config"] = {"workload": name,
                          "layers": [it["spec"].name for it in step.items],
                          "batch": step.items[0]["spec"].N,
                          "plans": [it["info"]["cand"] for it in step.items],
                          "l2": "flushed between steps (512 MB write, 512 MB read)"}
        # per-layer device time from the marks recorded after each layer
        layer_ms = [0.0] * len(step.items)
        starts = [a for a, _ in evs]
        per_step = len(step.items)
        for s_i in range(args.steps):
            prev = starts[s_i]
            for j in range(per_step):
                _, ev = marks[s_i * per_step + j]
                layer_ms[j] += prev.elapsed_time(ev)
                prev = ev
        per_layer = []
        for it, ms in zip(step.items, layer_ms):
            s = it["spec"]
            tpk, src = pipe_peak(peaks, s.in_dtype, it["info"]["kind"])
            t_flop = conv_flops(s) / (tpk * 1e12)
            t_byte = conv_bytes(s) / (peaks["hbm"] * 1e9)
            t = ms / args.steps / 1e3
            per_layer.append({"layer": s.name, "plan": it["info"]["cand"],
                              "us": t * 1e6, "tflops": conv_flops(s) / t / 1e12,
                              "roofline_us": max(t_flop, t_byte) * 1e6,
                              "roofline_frac": max(t_flop, t_byte) / t,
                              "bound": ("tensor" if it["info"]["kind"] == "umma" else "alu")
                              if t_flop >= t_byte else "hbm"})
        line["per_layer"] = per_layer
        # the whole step against its roofline: the sum of the layers' roofline times
        line["step_roofline_frac"] = (sum(p["roofline_us"] for p in per_layer) / 1e3
                                      / ms_per_step)
        if prof:
            dominant = max(prof.items(), key=lambda kv: kv[1][1])[0]
            line["roofline"] = kernel_roofline(dominant, prof, step, peaks, args, name)
        line["kernels"] = {k: {"launches": v[0], "ms": v[1]} for k, v in prof.items()}
    line["_specs"] = None if name == "bcast" else step.specs
    del step
    torch.cuda.empty_cache()
    return line


def synth_bcast_general():
    from broadcast_implicit_gemm_gb300 import synth
    return synth.BCAST_GENERAL


def bcast_var_dev(P, device):
    from broadcast_implicit_gemm_gb300 import synth
    return synth.bcast_var(P, seed=1).to(device)


HEADLINE = "resnet50_fp16"
# The other workloads, measured after the headline in the default run and
# reported under "workloads" on the same line.
EXTRAS = ["fused", "bcast", "depthwise_fp16", "sweep_fp32", "resnet_last"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=HEADLINE,
                    choices=["sweep_fp32", "resnet_last", "resnet50_fp16", "fused",
                             "depthwise_fp16", "bcast"])
    ap.add_argument("--only", action="store_true",
                    help="measure the named workload alone (no other workloads on the line)")
    ap.add_argument("--layer", default=None, help="run only the named layer of the workload")
    ap.add_argument("--no-search", action="store_true", help="heuristic plans, no timed search")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (smaller cases for profiling; "
                         "the line's config records it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local, dist = dist_setup(args)
    if args.impl == "reference":
        rc = run_reference(args, world, rank)
        if dist:
            dist.destroy_process_group()
        return rc

    import torch

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    flush = L2Flush(torch, device)
    peaks = load_peaks()

    head = measure(args.workload, args, device, stream, flush, peaks, world, dist, local)
    specs = head.pop("_specs")
    line = {
        "metric": METRIC, "value": head.pop("value"), "unit": head.pop("unit"), "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head.pop("ms_per_step"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "data": "synthetic",
    }
    line.update(head)
    extras = []
    if not (args.only or args.layer or args.batch) and args.workload == HEADLINE:
        extras = EXTRAS
    if extras:
        line["workloads"] = {}
        for name in extras:
            w = measure(name, args, device, stream, flush, peaks, world, dist, local)
            w.pop("_specs")
            line["workloads"][name] = w
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, specs)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
