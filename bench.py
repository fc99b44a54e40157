#!/usr/bin/env python
"""Benchmark of the FlashAttention backward (fa_bwd: preprocess + main + convert).

One step = one fa_bwd call over one batch of the workload (default: the GQA causal
workload B=4, Sq=Sk=2048, H=32, Hk=8, D=128), inputs resident in HBM, L2 flushed
between steps outside the timed events (a 256 MiB write, then a 256 MiB read that
writes the flush's dirty lines back, so each step starts on a cold, clean L2).  Prints
one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
  python bench.py --varlen [--workload NAME]   (packed sequences of mixed lengths; own line)
  python bench.py --block-density 0.5 [--workload NAME]   (block-sparse; own line)

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample of the
same workload (one batch x one kv-head group per step).  Under torchrun (N > 1) every
rank runs an independent replica (the path shards over (batch, kv-head) units with no
exchange); value = work of all ranks / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention-backward TFLOP/s (bf16) and % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = ("flushed between steps outside the timed events: 256 MiB write, then a 256 MiB "
           "read that writes the dirty lines back (cold, clean L2 at each step)")


class L2Flush:
    """Writes a buffer larger than L2 (evicting every line the previous step left), then
    reads a second one, so that the flush's own dirty lines are written back before the
    timed region instead of during it."""

    def __init__(self, device):
        import torch
        self.wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.rbuf = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.wbuf.zero_()
        self.rbuf.sum()


def link_bandwidth(device, nbytes=256 << 20, reps=5):
    """Pinned host <-> device copy bandwidth (GB/s) measured with CUDA events: host to
    device alone, device to host alone, and both at once on two streams (total bytes of
    both directions over the time of both)."""
    import torch
    h_src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_dst = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s1, s2 = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def timed(fn):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s1)
            s2.wait_event(e0)
            fn()
            s1.wait_stream(s2)
            e1.record(s1)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            d_a.copy_(h_src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_dst.copy_(d_b, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_in, t_out, t_both = timed(h2d), timed(d2h), timed(both)
    return {"h2d_gbs": round(nbytes / (t_in * 1e-3) / 1e9, 1),
            "d2h_gbs": round(nbytes / (t_out * 1e-3) / 1e9, 1),
            "both_gbs": round(2 * nbytes / (t_both * 1e-3) / 1e9, 1),
            "bytes_each_way": nbytes}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws_, device="cpu"):
    """The largest x over all ranks (a job's time is that of its slowest rank); x itself
    on a single process.  Collective: every rank must call it."""
    if ws_ <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step, steps, ws_, total_ms):
    """Whole-job throughput: the work every rank did (each rank runs its own replica of
    the workload) over the slowest rank's time."""
    return flops_per_step * steps * ws_ / (total_ms * 1e-3) / 1e12


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


KERNEL_SOURCES = {
    "fa_bwd_main": ("fa_bwd_main.cu", "fa_bwd_common.cuh", "fa_ptx.cuh", "fa_kernels.h", "fa_tiles.h"),
    "fa_bwd_wide": ("fa_wide.cu", "fa_bwd_common.cuh", "fa_ptx.cuh", "fa_kernels.h", "fa_tiles.h"),
}


def _kernel_source_hash(kernel="fa_bwd_main"):
    """Hash of a backward kernel's sources with comments and whitespace removed, so that
    the committed DRAM-traffic capture stays valid across comment-only edits."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "flashattention_backward_pass_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def _traffic(workload, kernel="fa_bwd_main"):
    """DRAM bytes per main-kernel launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", f"{kernel}.{workload}.traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") == _kernel_source_hash(kernel):
            return d.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        # samples taken while the GPU was busy: those at the highest power draw half
        pw = [num(r[3]) or 0.0 for r in rows]
        thr = sorted(pw)[len(pw) // 2] if pw else 0.0
        busy = [num(r[1]) for r, p in zip(rows, pw) if p >= thr and num(r[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(busy or sm) if (busy or sm) else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def run_ours(args, ws_, rank, local):
    import torch
    import flashattention_backward_pass_gb300 as fa
    from flashattention_backward_pass_gb300 import _abi
    from flashattention_backward_pass_gb300.workloads import ALL_WORKLOADS, make_inputs

    w = ALL_WORKLOADS[args.workload]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.load()
    q, k, v, do = make_inputs(w, dev)
    out, lse = fa.attention_forward(q, k, v, w.scale, w.causal, w.window_left, w.window_right,
                                    w.softcap)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsp = fa.alloc_bwd_workspace(q, k, args.deterministic, v)
    flush = L2Flush(dev)
    # The timed pass runs without the library's per-kernel events: an event between the
    # main and convert kernels would keep the convert kernel from starting on the SMs
    # the main kernel leaves.  The per-kernel split comes from a separate pass below.
    _abi.profile_enable(False)
    stream = torch.cuda.current_stream()

    def step():
        fa.fa_bwd(do, q, k, v, out, lse, dq, dk, dv, w.scale, w.causal, w.window_left,
                  w.window_right, w.softcap, args.deterministic, wsp)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(wsp) == 0

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    if ws_ > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if ws_ > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    status = fa.fa_bwd_status(wsp)
    # per-kernel split (events between the kernels; the convert kernel then runs after the
    # main kernel instead of overlapping its tail)
    _abi.profile_enable(True)
    main_ms, pre_ms, conv_ms = [], [], []
    for i in range(min(args.steps, 20)):
        flush()
        step()
        a, b_, c = _abi.profile_read()
        pre_ms.append(a)
        main_ms.append(b_)
        conv_ms.append(c)
    torch.cuda.synchronize()
    _abi.profile_enable(False)
    total_ms = max_over_ranks(total_ms, ws_, dev)

    # End to end through the public API with host buffers (pinned), copies in the region:
    # each step copies its inputs host -> device, runs fa_bwd and reads dq, dk, dv back.
    # The three stages run on their own streams with two device copies of the inputs and
    # outputs, so step k's compute overlaps step k+1's upload and step k-1's download, as a
    # caller that streams batches would run it.  Splitting the upload over two streams
    # measured the same: host <-> device bandwidth, not a copy engine, bounds it.
    e2e = None
    if not args.no_e2e:
        host_in = [x.cpu().pin_memory() for x in (do, q, k, v, out, lse)]
        host_out = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (dq, dk, dv)]
                    for _ in range(2)]
        dev_in = [[torch.empty_like(x) for x in (do, q, k, v, out, lse)] for _ in range(2)]
        dev_out = [[torch.empty_like(x) for x in (dq, dk, dv)] for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in host_in)
        d2h = sum(x.numel() * x.element_size() for x in host_out[0])
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        n_e2e = max(3, min(args.steps, 20))

        def e2e_step(it):
            j = it & 1
            if it >= 2:
                s_in.wait_event(done[j])        # step it-2 has finished reading dev_in[j]
                stream.wait_event(out_done[j])  # and its results in dev_out[j] are home
            with torch.cuda.stream(s_in):
                for dsrc, hsrc in zip(dev_in[j], host_in):
                    dsrc.copy_(hsrc, non_blocking=True)
                in_ready[j].record(s_in)
            stream.wait_event(in_ready[j])
            fa.fa_bwd(*dev_in[j], *dev_out[j], w.scale, w.causal, w.window_left, w.window_right,
                      w.softcap, args.deterministic, wsp, stream=stream)
            done[j].record(stream)
            s_out.wait_event(done[j])
            with torch.cuda.stream(s_out):
                for hdst, dsrc in zip(host_out[j], dev_out[j]):
                    hdst.copy_(dsrc, non_blocking=True)
                out_done[j].record(s_out)

        for it in range(2):
            e2e_step(it)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for it in range(2, 2 + n_e2e):
            e2e_step(it)
        for j in range(2):
            s_out.wait_event(out_done[j])
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws_, dev) / n_e2e
        # the host link's ceiling for this schedule: with upload, compute and download
        # overlapped, a step takes at least the longest of the three (each direction at
        # its own bandwidth, and both directions together at the concurrent bandwidth)
        link = link_bandwidth(dev)
        floor_ms = max(h2d / (link["h2d_gbs"] * 1e9) * 1e3, d2h / (link["d2h_gbs"] * 1e9) * 1e3,
                       (h2d + d2h) / (link["both_gbs"] * 1e9) * 1e3, total_ms / args.steps)
        e2e = {"value": round(job_tflops(w.nominal_flops, 1, ws_, e2e_ms), 3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 4),
               "schedule": "upload, fa_bwd and download on three streams, double-buffered",
               "link": link,
               "ceiling": {"ms_per_step": round(floor_ms, 4),
                           "value": round(job_tflops(w.nominal_flops, 1, ws_, floor_ms), 3),
                           "frac": round(floor_ms / e2e_ms, 4),
                           "note": "max(upload at h2d_gbs, download at d2h_gbs, both at "
                                   "both_gbs, the device-timed step)"}}

    # the forward that produces O and LSE (not part of the step): timed alone, L2 flushed
    fwd_ms = []
    for i in range(3 + min(args.steps, 20)):
        flush()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        fa.fa_fwd(q, k, v, out, lse, w.scale, w.causal, w.window_left, w.window_right, w.softcap)
        f1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            fwd_ms.append(f0.elapsed_time(f1))

    peaks, peak_src = _peaks()
    ms_per_step = total_ms / args.steps
    value = job_tflops(w.nominal_flops, args.steps, ws_, total_ms)
    main_avg = statistics.mean(main_ms)
    achieved = w.algorithmic_flops / (main_avg * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    wide = w.D != w.dv or w.D > 128
    main_kernel = "fa::bwd_wide_kernel" if wide else "fa::bwd_main_kernel"
    fwd_kernel = "fa::fwd_wide_kernel" if wide else "fa::fwd_tc_kernel"
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws_,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 inputs of the workload's shape)",
        "config": dict(w.describe(), deterministic=bool(args.deterministic),
                       l2=L2_NOTE,
                       parallelism=f"replicas x{ws_}" if ws_ > 1 else "single GPU",
                       flop_convention="10*B*H*Sq*Sk*D (2*(3D+2Dv) for Dv != D), halved for causal"),
        "pct_of_bf16_peak": round(100 * value / ws_ / peak, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": _traffic(args.workload, "fa_bwd_wide" if wide else "fa_bwd_main"),
                     "kernel": main_kernel,
                     "flops_per_launch": w.algorithmic_flops,
                     "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "frac_of_sustained": round(achieved / float(peaks["bf16_tflops_sustained"]), 4)},
        "kernel_ms": {"preprocess": round(statistics.mean(pre_ms), 4), "main": round(main_avg, 4),
                      "convert": round(statistics.mean(conv_ms), 4)},
        "forward": {"kernel": fwd_kernel, "ms": round(statistics.median(fwd_ms), 4),
                    "flops_per_launch": w.forward_flops,
                    "achieved_tflops": round(w.forward_flops
                                             / (statistics.median(fwd_ms) * 1e-3) / 1e12, 2),
                    "frac_of_peak": round(w.forward_flops
                                          / (statistics.median(fwd_ms) * 1e-3) / 1e12 / peak, 4),
                    "note": "fa_fwd (O, LSE) timed alone between L2 flushes; 2*(D + Dv) flops "
                            "per visible pair; not part of the timed step"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "device_status": status,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    return res


def _oracle_sample(w, b, hk, q, k, v, do):
    import numpy as np
    from oracle import attention_backward
    G = w.H // w.Hk
    hs = slice(hk * G, hk * G + G)
    f = lambda t: np.asarray(t, dtype=np.float64)
    attention_backward(f(do[b:b + 1, :, hs]), f(q[b:b + 1, :, hs]), f(k[b:b + 1, :, hk:hk + 1]),
                       f(v[b:b + 1, :, hk:hk + 1]), w.scale, causal=w.causal,
                       window_left=w.window_left, window_right=w.window_right, softcap=w.softcap)
    return w.nominal_flops / (w.B * w.Hk)


def cpu_baseline(w, budget_s=15.0):
    """The fp64 oracle, as it stands, on this host's cores: (batch, kv-head group) slices
    of the workload until about `budget_s` seconds of work."""
    from flashattention_backward_pass_gb300.workloads import make_inputs
    q, k, v, do = (t.float().numpy() for t in make_inputs(w, "cpu"))
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    flops, n = 0.0, 0
    t0 = time.perf_counter()
    while True:
        b, hk = divmod(n % (w.B * w.Hk), w.Hk)
        flops += _oracle_sample(w, b, hk, q, k, v, do)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} slice(s) of 1 batch x 1 kv-head group ({w.H // w.Hk} q-heads) of "
                      f"{w.name}, fp64 NumPy, {dt:.1f} s", "seconds": round(dt, 2)}


def run_reference(args, ws_, rank):
    from flashattention_backward_pass_gb300.workloads import ALL_WORKLOADS, make_inputs
    w = ALL_WORKLOADS[args.workload]
    q, k, v, do = (t.float().numpy() for t in make_inputs(w, "cpu"))
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    for i in range(args.warmup):
        b, hk = divmod(i % (w.B * w.Hk), w.Hk)
        _oracle_sample(w, b, hk, q, k, v, do)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        b, hk = divmod(i % (w.B * w.Hk), w.Hk)
        flops += _oracle_sample(w, b, hk, q, k, v, do)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"each step: the fp64 oracle backward on 1 batch x 1 kv-head group "
              f"({w.H // w.Hk} q-heads) of {w.name}")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(w.describe()),
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


VARLEN_MIX = (0.375, 0.25, 0.125, 0.125, 0.0625, 0.03125, 0.03125)


def _mix(total):
    lens = [int(total * f) for f in VARLEN_MIX]
    lens[0] += total - sum(lens)
    return lens


def run_varlen(args, ws_, local):
    """fa_bwd_varlen over the workload's tokens packed as sequences of mixed lengths
    (VARLEN_MIX of B*Sq query and B*Sk key rows; each sequence its own bottom-right mask)."""
    import torch
    import flashattention_backward_pass_gb300 as fa
    from flashattention_backward_pass_gb300 import _abi
    from flashattention_backward_pass_gb300.workloads import WORKLOADS, Workload, make_varlen_inputs

    w = WORKLOADS[args.workload]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.load()
    lq, lk = _mix(w.B * w.Sq), _mix(w.B * w.Sk)
    q, k, v, do, cu_q, cu_k = make_varlen_inputs(lq, lk, w.H, w.Hk, w.D, seed=w.seed, device=dev,
                                                 do_std=w.do_std)
    kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right,
              softcap=w.softcap)
    mq, mk = max(lq), max(lk)
    out, lse = fa.attention_forward_varlen(q, k, v, cu_q, cu_k, mq, mk, w.scale, **kw)
    dq, dk, dv = torch.empty_like(q), torch.zeros_like(k), torch.zeros_like(v)
    wsp = torch.empty(fa.bwd_varlen_workspace_size(len(lq), w.H, q.shape[0], w.D, args.deterministic),
                      dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    seqs = [Workload("seq", 1, a, b, w.H, w.Hk, w.D, w.causal, w.window_left, w.window_right,
                     w.softcap) for a, b in zip(lq, lk)]
    nominal = sum(x.nominal_flops for x in seqs)
    algorithmic = sum(x.algorithmic_flops for x in seqs)

    def step():
        fa.fa_bwd_varlen(do, q, k, v, out, lse, dq, dk, dv, cu_q, cu_k, mq, mk, w.scale,
                         deterministic=args.deterministic, workspace=wsp, **kw)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(wsp) == 0
    ms = []
    for _ in range(args.steps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    status = fa.fa_bwd_status(wsp)
    _abi.profile_enable(True)
    split = []
    for _ in range(min(args.steps, 20)):
        flush()
        step()
        split.append(_abi.profile_read())
    _abi.profile_enable(False)
    fwd = []
    for _ in range(min(args.steps, 20)):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fa.fa_fwd_varlen(q, k, v, out, lse, cu_q, cu_k, mq, mk, w.scale, **kw)
        e1.record(stream)
        torch.cuda.synchronize()
        fwd.append(e0.elapsed_time(e1))
    t = sum(ms) / len(ms)
    main_ms = statistics.mean(x[1] for x in split)
    peaks, _ = _peaks()
    return {"metric": METRIC, "value": round(nominal / (t * 1e-3) / 1e12, 3), "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16, packed sequences)",
            "config": dict(w.describe(), workload=w.name + "+varlen", lengths_q=lq, lengths_k=lk,
                           deterministic=bool(args.deterministic),
                           l2=L2_NOTE,
                           flop_convention="per sequence 10*H*Sq*Sk*D, halved for causal"),
            "main_kernel": {"ms": round(main_ms, 4),
                            "achieved_tflops": round(algorithmic / (main_ms * 1e-3) / 1e12, 2),
                            "frac_of_peak": round(algorithmic / (main_ms * 1e-3) / 1e12
                                                  / float(peaks["bf16_tflops"]), 4)},
            "kernel_ms": {"preprocess": round(statistics.mean(x[0] for x in split), 4),
                          "main": round(main_ms, 4),
                          "convert": round(statistics.mean(x[2] for x in split), 4)},
            "forward_ms": round(statistics.median(fwd), 4),
            "forward_tflops": round(0.4 * algorithmic / (statistics.median(fwd) * 1e-3) / 1e12, 2),
            "device_status": status}


def run_blocksparse(args, local):
    """fa_fwd_blocksparse + fa_bwd_blocksparse on the workload with a seeded random tile mask
    of the given density; value = 10*D flops per (query, key) pair left visible by the
    element mask and the tile mask together, per second of fa_bwd_blocksparse."""
    import numpy as np
    import torch
    import flashattention_backward_pass_gb300 as fa
    from flashattention_backward_pass_gb300 import _abi
    from flashattention_backward_pass_gb300.workloads import WORKLOADS, make_block_mask, make_inputs

    w = WORKLOADS[args.workload]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.load()
    q, k, v, do = make_inputs(w, dev)
    bm_cpu = make_block_mask(w.B, w.H, w.Sq, w.Sk, args.block_density, seed=w.seed)
    bm = bm_cpu.to(dev)
    kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right,
              softcap=w.softcap)
    # visible pairs: per (query tile, key tile) pair of the element mask, summed over kept pairs
    wr = 0 if w.causal else w.window_right
    i = np.arange(w.Sq)[:, None]
    j = np.arange(w.Sk)[None, :]
    vis = np.ones((w.Sq, w.Sk), dtype=bool)
    if wr >= 0:
        vis &= j <= i + (w.Sk - w.Sq) + wr
    if w.window_left >= 0:
        vis &= j >= i + (w.Sk - w.Sq) - w.window_left
    Mb, Nb = bm_cpu.shape[2], bm_cpu.shape[3]
    pad = np.zeros((Mb * 128, Nb * 128), dtype=np.int64)
    pad[:w.Sq, :w.Sk] = vis
    per_tile = pad.reshape(Mb, 128, Nb, 128).sum(axis=(1, 3))
    pairs = float((bm_cpu.numpy().astype(np.int64) * per_tile[None, None]).sum())
    flops = 10.0 * w.D * pairs
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.Sq, dtype=torch.float32, device=dev)
    fa.fa_fwd_blocksparse(q, k, v, out, lse, bm, w.scale, **kw)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsp = torch.empty(fa.bwd_blocksparse_workspace_size(w.B, w.H, w.Hk, w.Sq, w.Sk, w.D),
                      dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        ms = []
        for i in range(args.warmup + args.steps):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                ms.append(e0.elapsed_time(e1))
        return sum(ms) / len(ms)

    t = timed(lambda: fa.fa_bwd_blocksparse(do, q, k, v, out, lse, dq, dk, dv, bm, w.scale,
                                            workspace=wsp, deterministic=args.deterministic, **kw))
    status = fa.fa_bwd_status(wsp)
    tf = timed(lambda: fa.fa_fwd_blocksparse(q, k, v, out, lse, bm, w.scale, **kw))
    peaks, _ = _peaks()
    return {"metric": METRIC, "value": round(flops / (t * 1e-3) / 1e12, 3), "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16, seeded random tile mask)",
            "config": dict(w.describe(), workload=w.name + "+blocksparse",
                           block_density=args.block_density,
                           deterministic=bool(args.deterministic),
                           kept_tile_pairs=int(bm_cpu.sum()),
                           l2=L2_NOTE,
                           flop_convention="10*D per visible (query, key) pair after both masks"),
            "pct_of_bf16_peak": round(100 * flops / (t * 1e-3) / 1e12 / float(peaks["bf16_tflops"]), 2),
            "forward_ms": round(tf, 4),
            "forward_tflops": round(0.4 * flops / (tf * 1e-3) / 1e12, 2),
            "device_status": status}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gqa_causal",
                    help="one of the five workloads (default: the GQA causal headline), or "
                         "gqa_causal_d256 / gqa_causal_d192_dv128 (the wide kernels)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--deterministic", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--varlen", action="store_true",
                    help="time fa_bwd_varlen on the workload's tokens packed as a length mix "
                         "(a separate line, not the headline)")
    ap.add_argument("--block-density", type=float, default=None,
                    help="time fa_bwd_blocksparse with a random tile mask of this density "
                         "(a separate line, not the headline)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    ws_, rank, local = _dist()

    if args.block_density is not None:
        if rank == 0:
            print(json.dumps(run_blocksparse(args, local)), flush=True)
        return
    if args.varlen:
        if rank == 0:
            print(json.dumps(run_varlen(args, ws_, local)), flush=True)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, ws_, rank)), flush=True)
        return

    if ws_ > 1:
        import torch
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, ws_, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws_ > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
