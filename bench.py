#!/usr/bin/env python
"""Benchmark of the conv3d / conv_transpose3d hot path on GB300.

One step = one forward call of each of the four full-size workloads
(Conv3d (3,3,1) [16,16,128,128,8]->64; ConvTranspose3d 32->64 k3 s2 p1 d2 on
[16,32,16,32,32]; ConvTranspose3d 3->16 + BatchNorm3d + 4x4x4 avg pool on
[64,3,32,32,32]; Conv3d 32->64 k3 p1 + MaxPool3d(2) + channel logsumexp + ReLU
on [4,32,32,128,128]).  These cover every step of the path: validation and
planning, weight packing, TMA staging, the 3xTF32 tensor-core main loop and
the three fused epilogues with the BatchNorm finalize.

Metric: effective TFLOP/s = 2 x valid MACs (taps whose input index is in
range) / device time, results fp32-accurate (1e-4 against the fp64 oracle).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  The L2 cache is flushed (a 256 MB write)
before every timed call; calls are timed with CUDA events on the stream the
library launches on.  --impl reference times the fp64 CPU oracle on bounded
samples of the same workloads on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from transposed_conv_epilogues_gb300 import workloads as W  # noqa: E402

BENCH_WORKLOADS = ["conv331", "convT_s2p1d2", "convT_bn_avgpool", "conv_maxpool_lse_relu"]
# the tiny (3,3,1) conv is launch-bound: its ms is reported beside the step,
# outside the aggregate
REPORTED_ONLY = ["conv331_tiny"]
TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense tensor-core rate ratio (GB300)


def peaks():
    """(hbm GB/s, bf16 TFLOP/s, source) from the measured peaks file."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def measure_tf32_peak(dev):
    """Dense TF32 tensor-core throughput of this GPU, TFLOP/s: cuBLAS fp32
    GEMMs with TF32 enabled (8192^3 and 16384^3, best of 10 each, CUDA
    events), the larger of the two.  The fp32-accurate (3xTF32) peak is a
    third of it."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    best = 0.0
    try:
        for n in (8192, 16384):
            a = torch.randn(n, n, device=dev)
            b = torch.randn(n, n, device=dev)
            for _ in range(3):
                c = a @ b
            torch.cuda.synchronize(dev)
            for _ in range(10):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                c = a @ b
                e1.record()
                torch.cuda.synchronize(dev)
                best = max(best, 2.0 * n ** 3 / (e0.elapsed_time(e1) * 1e-3) / 1e12)
            del a, b, c
        torch.cuda.empty_cache()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return best


def max_over_ranks(values, world, device):
    """Element-wise max of a list of floats over the ranks of the process
    group (identity on one rank): each rank's time reduced to the job's."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.gpu_id], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [t.strip() for t in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


# the sources each captured kernel is built from (a capture stays valid while
# they are unchanged)
KERNEL_SOURCES = {
    "engine": ["engine.cu", "engine.cuh", "fill.cuh", "ptx.cuh", "plan.h", "plan.cpp"],
    "lag": ["lag.cu", "pool.cuh", "ptx.cuh", "plan.h", "plan.cpp"],
    "pooled": ["pool.cu", "pool.cuh", "ptx.cuh", "plan.h", "plan.cpp"],
    "direct": ["direct.cu", "direct.cuh", "plan.h", "plan.cpp"],
}


def source_hash(kind="engine"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "transposed_conv_epilogues_gb300", "csrc")
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_by_workload.txt")
    try:
        with open(path) as f:
            t = json.load(f)
    except Exception:
        return None
    e = t.get(kernel_workload)
    if not e or e.get("sources", "engine") not in KERNEL_SOURCES:
        return None
    if e.get("source_hash") != source_hash(e.get("sources", "engine")):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle on bounded samples (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
ORACLE_SAMPLES = {"conv331": 20000000, "convT_s2p1d2": 6000000, "convT_bn_avgpool": 20000000,
                  "convT_bneval_avgpool": 20000000, "dwconv_k3": 20000000,
                  "dwconv_k3_ndhwc": 20000000, "conv_k3_ndhwc": 2000000,
                  "conv_maxpool_lse_relu": 2000000}


def oracle_sample_run(names, scale=1.0, inputs_cache=None):
    """Time the oracle's core operator on sampled outputs of each workload.
    Returns (valid flops done, seconds, threads, description)."""
    import numpy as np

    import oracle
    from transposed_conv_epilogues_gb300 import inputs
    oracle.build()
    threads = os.cpu_count() or 1
    flops = 0.0
    secs = 0.0
    desc = []
    for n in names:
        wl = W.BY_NAME[n]
        if inputs_cache is not None and n in inputs_cache:
            x, w, b = inputs_cache[n]
        else:
            x, w, b = wl.make_inputs()
            if inputs_cache is not None:
                inputs_cache[n] = (x, w, b)
        O = W.out_spatial(wl)
        total = wl.x_shape[0] * wl.cout * int(np.prod(O))
        cnt = max(1, int(ORACLE_SAMPLES.get(n, 2000000) * scale))
        idx = inputs.sample_indices(9000 + wl.index, total, cnt)
        kw = dict(stride=wl.stride, padding=wl.padding, dilation=wl.dilation, groups=wl.groups)
        t0 = time.perf_counter()
        if wl.transposed:
            oracle.conv_transpose3d_at(x, w, b, idx, output_padding=wl.output_padding,
                                       nthreads=threads, **kw)
        else:
            oracle.conv3d_at(x, w, b, idx, nthreads=threads, **kw)
        secs += time.perf_counter() - t0
        flops += 2.0 * W.valid_macs(wl) / total * len(idx)
        desc.append(f"{n}: {len(idx)} outputs")
    return flops, secs, threads, "oracle core operator (fp64) on sampled outputs; " + "; ".join(
        desc)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from transposed_conv_epilogues_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    import transposed_conv_epilogues_gb300 as tc
    tc.load()

    hbm, bf16_peak, peak_src = peaks()
    tf32_measured = measure_tf32_peak(dev)
    tf_peak = tf32_measured / 3.0  # fp32-accurate products: three TF32 MMAs each
    tf_peak_derived = bf16_peak * TF32_OVER_BF16 / 3.0
    names = args.workloads.split(",")
    extra = [n for n in REPORTED_ONLY if n not in names] if names == BENCH_WORKLOADS else []
    wls = [W.BY_NAME[n] for n in names + extra]
    host = {n: W.BY_NAME[n].make_inputs() for n in names + extra}
    # evaluation-mode BatchNorm: running mean / variance, gamma, beta
    host_bn = {wl.name: wl.make_bn_eval_params() for wl in wls
               if wl.op == "convT_bneval_avgpool"}
    dev_in = {}
    host_call = {}  # inputs in the layout of the call (the oracle keeps NCDHW)
    dev_bn = {n: tuple(torch.from_numpy(a).to(dev) for a in v) for n, v in host_bn.items()}
    outs = {}
    for wl in wls:
        x, w, b = host[wl.name]
        if wl.op == "conv3d_ndhwc":  # the same values, channels-last
            x = np.ascontiguousarray(x.transpose(0, 2, 3, 4, 1))
        host_call[wl.name] = (x, w, b)
        dev_in[wl.name] = tuple(None if a is None else torch.from_numpy(a).to(dev)
                                for a in (x, w, b))
        outs[wl.name] = torch.empty(W.y_shape(wl), dtype=torch.float32, device=dev)

    op_of = {"conv3d": 0, "conv_transpose3d": 1, "conv_maxpool_lse_relu": 2,
             "convT_bn_avgpool": 3, "convT_bneval_avgpool": 4, "conv3d_ndhwc": 5}
    wss = {}
    for wl in wls:
        nb = tc.workspace_bytes(op_of[wl.op], wl.x_shape, wl.w_shape, wl.stride, wl.padding,
                                wl.dilation, wl.output_padding, wl.groups)
        wss[wl.name] = torch.empty(nb, dtype=torch.uint8, device=dev)

    def call(wl, x, w, b, out, bn=None):
        kw = dict(stride=wl.stride, padding=wl.padding, dilation=wl.dilation, groups=wl.groups,
                  out=out, workspace=wss[wl.name])
        if wl.op == "conv3d":
            return tc.conv3d_fwd(x, w, b, **kw)
        if wl.op == "conv3d_ndhwc":
            return tc.conv3d_fwd_ndhwc(x, w, b, **kw)
        if wl.op == "conv_transpose3d":
            return tc.conv_transpose3d_fwd(x, w, b, output_padding=wl.output_padding, **kw)
        if wl.op == "conv_maxpool_lse_relu":
            return tc.conv_maxpool_lse_relu(x, w, b, **kw)
        if wl.op == "convT_bneval_avgpool":
            rm, rv, g, be = bn if bn is not None else dev_bn[wl.name]
            return tc.convT_bneval_avgpool(x, w, b, rm, rv, g, be, wl.eps,
                                           output_padding=wl.output_padding, **kw)
        return tc.convT_bn_avgpool(x, w, b, None, None, wl.eps,
                                   output_padding=wl.output_padding, **kw)

    # library launches per call: weight pack + engine (the transposed conv's
    # bias fill runs inside the engine; + BatchNorm finalize and apply for
    # batch statistics; + the running-statistics affine for evaluation mode)
    # (the convT_bneval path: finalize + pack + pooled conv; grouped convs
    # with few channels per group: one direct launch; channels-last convs
    # the engine's channels-last mode does not take: transpose + pack +
    # engine + transpose)
    def launches(wl):
        if wl.op in ("conv3d", "conv3d_ndhwc"):
            pl = tc.plan_describe(op_of[wl.op], wl.x_shape, wl.w_shape, wl.stride, wl.padding,
                                  wl.dilation, wl.output_padding, wl.groups)
            if pl.get("direct"):
                return 1
            # channels-last outside the engine's channels-last mode: + the two
            # layout transposes
            return 4 if wl.op == "conv3d_ndhwc" and not pl.get("cl") else 2
        if wl.op in ("convT_bn_avgpool", "convT_bneval_avgpool"):
            pl = tc.plan_describe(op_of[wl.op], wl.x_shape, wl.w_shape, wl.stride, wl.padding,
                                  wl.dilation, wl.output_padding, wl.groups)
            if pl.get("pool_path"):
                # batch statistics: lag kernel + reduction + per-channel finalize,
                # or Gram + reduction + finalize; running statistics: finalize; then the
                # pooled conv (the direct kernel, or weight pack + engine)
                pooled = 1 if max(pl["pool_Ke"]) <= 3 and wl.x_shape[1] <= 4 else 2
                if wl.op == "convT_bneval_avgpool":
                    return 1 + pooled
                return 3 + pooled
            return 4 if wl.op == "convT_bn_avgpool" else 3
        return {"conv_transpose3d": 2, "conv_maxpool_lse_relu": 2}[wl.op]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = {wl.name: [] for wl in wls}

    # warm-up
    for _ in range(args.warmup):
        for wl in wls:
            call(wl, *dev_in[wl.name], outs[wl.name])
    torch.cuda.synchronize()
    if tc.last_device_error() != tc.TC3D_OK:
        raise RuntimeError("device error during warm-up")

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) == 36:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        for wl in wls:
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call(wl, *dev_in[wl.name], outs[wl.name])
            e1.record(stream)
            ev[wl.name].append((e0, e1))
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    if tc.last_device_error() != tc.TC3D_OK:
        raise RuntimeError("device error during the timed region")

    per = {}
    reported = {}
    step_ms = 0.0
    total_flops = 0.0
    # mean event time per workload, then the max over ranks
    mean_ms = max_over_ranks([sum(a.elapsed_time(b) for a, b in ev[wl.name]) / len(ev[wl.name])
                              for wl in wls], world, dev)
    for wl, ms in zip(wls, mean_ms):
        ts = [a.elapsed_time(b) for a, b in ev[wl.name]]
        fl = 2.0 * W.valid_macs(wl)
        by = W.algorithmic_bytes(wl)
        t_tc = fl / (tf_peak * 1e12)
        t_hbm = by / (hbm * 1e9)
        bound = "tensor" if t_tc >= t_hbm else "hbm"
        t_roof = max(t_tc, t_hbm)
        entry = {
            "ms": round(ms, 4), "ms_median": round(statistics.median(ts), 4),
            "tflops": round(fl / (ms * 1e-3) / 1e12, 3),
            "gbs": round(by / (ms * 1e-3) / 1e9, 1),
            "valid_gflop": round(fl / 1e9, 3), "dense_gflop": round(2.0 * W.dense_macs(wl) / 1e9, 3),
            "alg_mb": round(by / 1e6, 2), "bound": bound,
            "roofline_ms": round(t_roof * 1e3, 4), "roofline_frac": round(t_roof / (ms * 1e-3), 4),
        }
        if wl.name in extra:
            entry["note"] = "launch-bound; reported beside the step, not in the aggregate"
            reported[wl.name] = entry
            continue
        per[wl.name] = entry
        step_ms += ms
        total_flops += fl
    value = world * total_flops / (step_ms * 1e-3) / 1e12

    # dominant kernel: the workload with the longest call
    dom = max((w_ for w_ in wls if w_.name in per), key=lambda w_: per[w_.name]["ms"])
    pd = per[dom.name]
    if pd["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": pd["tflops"], "peak": round(tf_peak, 1),
                "unit": "TFLOP/s", "frac": round(pd["tflops"] / tf_peak, 4),
                "peak_source": "measured live: cuBLAS TF32 GEMM (best of 8192^3 and 16384^3, "
                               "best of 10 each) / 3 (3xTF32 passes)",
                "tf32_tflops_measured": round(tf32_measured, 1),
                "peak_derived_from_bf16": round(tf_peak_derived, 1)}
    else:
        roof = {"bound": "hbm", "achieved": pd["gbs"], "peak": hbm, "unit": "GB/s",
                "frac": round(pd["gbs"] / hbm, 4), "peak_source": f"{peak_src} copy bandwidth"}
    roof["kernel"] = f"engine_kernel ({dom.name})"
    roof["traffic"] = recorded_traffic(dom.name)

    # end to end through the public API with host buffers
    pinned_in = {}
    pinned_bn = {n: tuple(torch.from_numpy(a).pin_memory() for a in v)
                 for n, v in host_bn.items()}
    pinned_out = {}
    h2d = sum(a.numel() * 4 for v in pinned_bn.values() for a in v)
    d2h = 0
    step_wls = [w_ for w_ in wls if w_.name in per]
    # The host link bounds this measure (its device-to-host direction above
    # all: the step's results are 2.4 x its inputs), so the workloads go in
    # the order that starts the largest results earliest: by results per
    # input byte, largest first.  Every one still runs once per step.
    io_bytes = {}
    for wl in step_wls:
        nin = sum(int(np.prod(a.shape)) for a in host_call[wl.name] if a is not None)
        io_bytes[wl.name] = int(np.prod(W.y_shape(wl))) / max(1, nin)
    step_wls.sort(key=lambda w_: -io_bytes[w_.name])
    for wl in step_wls:
        pinned_in[wl.name] = tuple(None if a is None else torch.from_numpy(a).pin_memory()
                                   for a in host_call[wl.name])
        pinned_out[wl.name] = torch.empty(W.y_shape(wl), dtype=torch.float32).pin_memory()
        h2d += sum(a.numel() * 4 for a in pinned_in[wl.name] if a is not None)
        d2h += pinned_out[wl.name].numel() * 4
    e2e_steps = max(1, min(args.steps, 5))
    # Copies overlap the library calls as a caller would arrange them: the
    # inputs of each workload go in on one stream, the calls run on the
    # compute stream, the results come out on a third; events order each
    # workload's three stages, and across steps no device buffer is
    # refilled before the call that read it, or re-written before its
    # result was copied out.  Every step still moves all of its inputs in
    # and all of its results out inside its own timed region.
    # several copy streams per direction: large copies are split in chunks
    # over them, so that more than one copy engine moves them
    n_cp = 4
    s_in = torch.cuda.Stream(dev)
    s_outs = [torch.cuda.Stream(dev) for _ in range(n_cp)]

    def chunked_copy(dst, src, streams):
        d, s_ = dst.view(-1), src.view(-1)
        step = (d.numel() + len(streams) - 1) // len(streams)
        for i, st in enumerate(streams):
            lo, hi = i * step, min(d.numel(), (i + 1) * step)
            if lo < hi:
                with torch.cuda.stream(st):
                    d[lo:hi].copy_(s_[lo:hi], non_blocking=True)

    d_in = {n: tuple(None if a is None else torch.empty(a.shape, dtype=a.dtype, device=dev)
                     for a in v) for n, v in pinned_in.items()}
    d_bn = {n: tuple(torch.empty(a.shape, dtype=a.dtype, device=dev) for a in v)
            for n, v in pinned_bn.items()}
    ev_done = {}   # the call that last read a workload's input buffers
    ev_read = {}   # the copy that last read a workload's output buffer
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e2e_ms = []
    # untimed warm-up steps of the same sequence first (first use of the copy
    # streams and of the pinned buffers), as for the device-timed steps
    e2e_warm = min(2, max(1, args.warmup))
    for it in range(e2e_warm + e2e_steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        for st in s_outs:
            st.wait_event(e0)
        for wl in step_wls:
            n = wl.name
            if n in ev_done:
                s_in.wait_event(ev_done[n])
            with torch.cuda.stream(s_in):
                for dst, src in zip(d_in[n], pinned_in[n]):
                    if src is not None:
                        dst.copy_(src, non_blocking=True)
                for dst, src in zip(d_bn.get(n, ()), pinned_bn.get(n, ())):
                    dst.copy_(src, non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(s_in)
            stream.wait_event(loaded)
            if n in ev_read:
                stream.wait_event(ev_read[n])
            call(wl, *d_in[n], outs[n], d_bn.get(n))
            done = torch.cuda.Event()
            done.record(stream)
            ev_done[n] = done
            for st in s_outs:
                st.wait_event(done)
            chunked_copy(pinned_out[n], outs[n], s_outs)
            for st in s_outs[1:]:
                s_outs[0].wait_stream(st)
            read = torch.cuda.Event()
            read.record(s_outs[0])
            ev_read[n] = read
        stream.wait_stream(s_in)
        for st in s_outs:
            stream.wait_stream(st)
        e1.record(stream)
        torch.cuda.synchronize()
        if it >= e2e_warm:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e = max_over_ranks([statistics.mean(e2e_ms)], world, dev)[0]

    line = {
        "metric": "effective TFLOP/s (2 x valid MACs / device time), fp32-accurate (1e-4 vs "
                  "fp64 oracle), four full-size workloads per step",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "tf32x3",
        "data": "synthetic: seeded splitmix64, x ~ N(0,1), w and bias ~ U(+-1/sqrt(fan_in))",
        "config": {
            "workload": "+".join(names) + (" (the four full-size configs, one call each)"
                                           if names == BENCH_WORKLOADS else " (one call each)"),
            "per_workload": per,
            "reported_only": reported,
            "peaks": {"hbm_gbs": hbm, "hbm_source": f"{peak_src} copy bandwidth",
                      "tf32_tflops_measured": round(tf32_measured, 1),
                      "tf32x3_tflops": round(tf_peak, 1)},
            "l2": "flushed by a 256 MB device write before every timed call",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "wall_s_timed_region": round(wall, 3),
        },
        "roofline": roof,
        "e2e": {"value": round(world * total_flops / (e2e * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * sum(launches(wl) for wl in wls),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # repeat the fixed output sample until about 10 s of oracle work ran
        fl = secs = 0.0
        reps = 0
        while reps < 40 and (secs < 10.0 or reps == 0):
            f1, s1, thr, desc = oracle_sample_run(names, inputs_cache=host)
            fl += f1
            secs += s1
            reps += 1
        line["cpu_baseline"] = {"value": round(fl / secs / 1e12, 6), "unit": "TFLOP/s",
                                "cores": thr, "kind": "oracle",
                                "sample": f"{reps} x ({desc})", "seconds": round(secs, 2)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    names = args.workloads.split(",")
    cache = {}
    scale = 0.005
    for _ in range(args.warmup):
        oracle_sample_run(names, scale=scale, inputs_cache=cache)
    tot_fl = tot_s = 0.0
    desc, thr = "", 1
    for _ in range(args.steps):
        fl, secs, thr, desc = oracle_sample_run(names, scale=scale, inputs_cache=cache)
        tot_fl += fl
        tot_s += secs
    value = tot_fl / tot_s / 1e12
    line = {
        "impl": "reference",
        "metric": "effective TFLOP/s (2 x valid MACs / device time), fp32-accurate (1e-4 vs "
                  "fp64 oracle), four full-size workloads per step",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * tot_s / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded splitmix64, x ~ N(0,1), w and bias ~ U(+-1/sqrt(fan_in))",
        "config": {"workload": "+".join(names) + " (bounded output samples per step)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": thr,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workloads", default=",".join(BENCH_WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
