"""Benchmark: block-sparse attention fwd+bwd at seq 8192 on GB300.

One step = bsr_attn_fwd + bsr_attn_bwd over one batch of synthetic inputs
(default workload: batch 1, heads 16, seq 8192, head_dim 128, bf16, block
mask = band |m-n| <= 2 plus block row 0 and block column 0, 436 stored
blocks).  Throughput is counted over stored blocks only: 4*128^2*D FLOP
forward and 10*128^2*D backward per stored block and head.

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]

Prints ONE JSON line on rank 0.  Multi-GPU runs (torchrun) are independent
replicas with the whole workload per rank (weak scaling); timing is the max
over ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from block_sparse_attention_bsr_gb300 import inputs  # noqa: E402

BLOCK = 128
METRIC = "fwd+bwd ms & TFLOP/s over stored blocks at seq 8192; % of GB300 bf16 TC peak"
# contraction FLOP per stored block and head, as each kernel executes them
# (x 128^2 * D).  The head_dim-64/128 dK/dV walk recomputes S and dP; on a
# plan the dQ walk sums the dS tiles it stored (dq_ds: dQ += dS K only), per
# call it recomputes S and dP as well (dq_tc); the wide kernels recompute the scores once per output slice
# of W columns (W = 256 for 16-bit operands, 128 for fp32) and run fp32 as six
# bf16 piece products, all counted here as the bf16 MMAs they issue.
FLOP_PER_BLOCK = {"fwd_tc": 4, "fwd2p_stats": 2, "fwd2p_out": 4, "dq_tc": 6, "dq_ds": 2, "dv_ps": 2, "dkdv_tc": 8}
WIDE_SCORE_MMAS = {"fwd_wide": 1, "dq_wide": 2, "dv_wide": 1, "dk_wide": 2}  # score contractions per slice


def alg_flops(wl, nnzb, part="total"):
    per = {"fwd": 4, "bwd": 10, "total": 14}[part]
    return per * BLOCK * BLOCK * wl.head_dim * nnzb * wl.batch * wl.heads


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of a
# kernel on a workload, from one ncu capture, with the SHA-256 of the source
# files the kernel was built from at the time; reported only while the
# current sources still hash the same (otherwise the roofline's traffic is
# null until the kernel is captured again).
MEASURED_TRAFFIC = {
    ("global_s8192", "fwd_tc"): {"bytes": 136.4e6, "sources": ("tc_fwd2.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "6b348a4d57aa31d13d83b62106bb1fe180754b6caba85bc0d31858b530f06bca"},
    ("global_s8192", "dkdv_tc"): {"bytes": 429.5e6, "sources": ("tc_bwd.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "f6edce16f7f0891c387bf9277bb89b8a8a71a150b47ac2839e4e0fecc62a5d89"},
    ("global_s8192", "dq_ds"): {"bytes": 300.3e6, "sources": ("tc_bwd.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "f6edce16f7f0891c387bf9277bb89b8a8a71a150b47ac2839e4e0fecc62a5d89"},
    ("local_s8192_d256", "fwd_wide"): {"bytes": 114.6e6, "sources": ("tc_wide.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "5fa2010596880ff8b1fab5eb3282367a0570e2874181c90e6333c03d1c77a5aa"},
    ("local_s8192_d256", "dk_wide"): {"bytes": 364.4e6, "sources": ("tc_wide.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "5fa2010596880ff8b1fab5eb3282367a0570e2874181c90e6333c03d1c77a5aa"},
    ("local_s8192_d256", "dq_ds"): {"bytes": 162.1e6, "sources": ("tc_bwd.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "f6edce16f7f0891c387bf9277bb89b8a8a71a150b47ac2839e4e0fecc62a5d89"},
    ("local_s8192_d256", "dv_ps"): {"bytes": 161.6e6, "sources": ("tc_bwd.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "f6edce16f7f0891c387bf9277bb89b8a8a71a150b47ac2839e4e0fecc62a5d89"},
    ("global_s8192_f32", "fwd_wide"): {"bytes": 526.3e6, "sources": ("tc_wide.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "5fa2010596880ff8b1fab5eb3282367a0570e2874181c90e6333c03d1c77a5aa"},
    ("global_s8192_f32", "dk_wide"): {"bytes": 1872.4e6, "sources": ("tc_wide.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "5fa2010596880ff8b1fab5eb3282367a0570e2874181c90e6333c03d1c77a5aa"},
    ("global_s8192_f32", "dq_ds"): {"bytes": 696.2e6, "sources": ("tc_wide.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "5fa2010596880ff8b1fab5eb3282367a0570e2874181c90e6333c03d1c77a5aa"},
    ("global_s8192_f32", "dv_ps"): {"bytes": 696.8e6, "sources": ("tc_wide.cu", "sm100.cuh", "sched.cuh"),
        "sha256": "5fa2010596880ff8b1fab5eb3282367a0570e2874181c90e6333c03d1c77a5aa"},
}


def measured_traffic(workload, kernel):
    rec = MEASURED_TRAFFIC.get((workload, kernel))
    if rec is None:
        return None
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "block_sparse_attention_bsr_gb300", "csrc")
    for f in rec["sources"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest() == rec["sha256"] else None


def kernel_flops(name, wl, nnzb):
    per_head = BLOCK * BLOCK * wl.head_dim * nnzb * wl.batch * wl.heads
    if name in ("dq_ds", "dv_ps") and wl.dtype == "f32":  # five bf16 piece products per product
        return 10 * per_head
    for key, mult in FLOP_PER_BLOCK.items():
        if name.startswith(key):
            return mult * per_head
    if name in WIDE_SCORE_MMAS:
        w = min(wl.head_dim, 128 if wl.dtype == "f32" else 256)
        nsl = max(1, wl.head_dim // w)
        f32 = wl.dtype == "f32"
        # fp32: six bf16 piece products per score product; the accumulate
        # products take six too, but five where P goes in two pieces (forward, dV)
        score_terms = 6 if f32 else 1
        acc_terms = (5 if name in ("fwd_wide", "dv_wide") else 6) if f32 else 1
        return (score_terms * 2 * WIDE_SCORE_MMAS[name] * nsl + acc_terms * 2) * per_head
    return None


def kernel_bytes(name, wl, nnzb):
    """Algorithmic DRAM bytes of one launch of a streaming kernel, else None: the dQ walk over stored dS
    tiles (dq_ds) reads every dS tile once (128 x 128 16-bit values per stored block and head), each head's
    K once and writes dQ once."""
    if name in ("dq_ds", "dv_ps"):  # dV over stored P^T tiles: the same stream
        e = 2
        return wl.batch * wl.heads * (nnzb * BLOCK * BLOCK * e + 2 * wl.seq * wl.head_dim * e)
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(bf16=d.get("bf16_tflops"), bf16_sustained=d.get("bf16_tflops_sustained"),
                    hbm=d.get("hbm_gbs"), source="measured")
    return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def flush_l2(buf):
    buf.add_(1)  # writes the whole buffer (larger than the 129 MB L2)


def run_ours(args, rank, world, dev):
    import block_sparse_attention_bsr_gb300 as bsr

    wl = inputs.WORKLOADS[args.workload]
    bm = wl.block_mask()
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, wl.nb, dev)
    nnzb = st.nnzb
    hQ, hK, hV, hdO = wl.inputs(seed=0)
    Q, K, V, dO = (t.to(dev) for t in (hQ, hK, hV, hdO))
    O = torch.empty_like(Q)
    rm = torch.empty(Q.shape[:3], device=dev, dtype=torch.float32)
    rd = torch.empty_like(rm)
    dQ, dK, dV = (torch.empty_like(Q) for _ in range(3))
    stream = torch.cuda.current_stream(dev)

    two_pass = args.forward == "two-pass"
    # The step runs on a reusable plan of the mask (bsr_plan_create, built once
    # here, outside the timed region: the work lists and scratch of a static
    # structure); --api per-call times the entry points that plan on every call.
    planned = args.api == "plan" and not two_pass
    plan = st.plan(Q) if planned else None

    def step(q, k, v, do, o, m, d, gq, gk, gv):
        if planned:
            bsr.bsr_attn_fwd_plan(plan, q, k, v, wl.scale, o, m, d, stream)
            bsr.bsr_attn_bwd_plan(plan, q, k, v, o, do, m, d, wl.scale, gq, gk, gv, stream)
            return
        bsr.bsr_attn_fwd(q, k, v, st.row_ptr, st.col_idx, st.n_brows, BLOCK, wl.scale, o, m, d, stream, two_pass)
        bsr.bsr_attn_bwd(q, k, v, o, do, m, d, st.row_ptr, st.col_idx, st.col_ptr, st.row_idx, wl.scale,
                         gq, gk, gv, stream)

    def step_per_call(q, k, v, do, o, m, d, gq, gk, gv):
        bsr.bsr_attn_fwd(q, k, v, st.row_ptr, st.col_idx, st.n_brows, BLOCK, wl.scale, o, m, d, stream, two_pass)
        bsr.bsr_attn_bwd(q, k, v, o, do, m, d, st.row_ptr, st.col_idx, st.col_ptr, st.row_idx, wl.scale,
                         gq, gk, gv, stream)

    args_dev = (Q, K, V, dO, O, rm, rd, dQ, dK, dV)
    l2 = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        flush_l2(l2)
        step(*args_dev)
    bsr.bsr_attn_check()

    # device-resident timed region: per-step CUDA events, L2 flushed before each step
    def timed_steps(per_kernel, nsteps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nsteps)]
        bsr.profile_collect()
        bsr.profile_enable(per_kernel)
        barrier(world)
        torch.cuda.synchronize(dev)
        for i in range(nsteps):
            flush_l2(l2)
            evs[i][0].record(stream)
            step(*args_dev)
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        bsr.profile_enable(False)
        prof = bsr.profile_collect()
        bsr.bsr_attn_check()
        ts = [a.elapsed_time(b) for a, b in evs]
        return (max_over_ranks(statistics.median(ts), world), max_over_ranks(sum(ts) / nsteps, world), prof)

    # The headline pass records no events between the kernels of a step (each
    # such record adds a few microseconds of idle GPU time); a second pass of
    # the same K steps brackets every launch with events for the per-kernel
    # durations the roofline uses.  The headline statistic is the median of
    # the K per-step times; a longer pass of 100 steps is reported beside it.
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        ms_per_step, ms_mean, _ = timed_steps(False, args.steps)
        ms_per_step_instr, _, prof = timed_steps(True, args.steps)
    long_steps = max(100, args.steps)
    ms_long, ms_long_mean, _ = timed_steps(False, long_steps)

    # forward alone and backward alone (same protocol, untimed for the headline)
    def time_part(fn, reps):
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i in range(reps):
            flush_l2(l2)
            e[i][0].record(stream)
            fn()
            e[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in e)

    if planned:
        ms_fwd = time_part(lambda: bsr.bsr_attn_fwd_plan(plan, Q, K, V, wl.scale, O, rm, rd, stream),
                           max(args.steps, 5))
        ms_bwd = time_part(lambda: bsr.bsr_attn_bwd_plan(plan, Q, K, V, O, dO, rm, rd, wl.scale, dQ, dK, dV,
                                                         stream), max(args.steps, 5))
    else:
        ms_fwd = time_part(lambda: bsr.bsr_attn_fwd(Q, K, V, st.row_ptr, st.col_idx, st.n_brows, BLOCK, wl.scale,
                                                     O, rm, rd, stream, two_pass), max(args.steps, 5))
        ms_bwd = time_part(lambda: bsr.bsr_attn_bwd(Q, K, V, O, dO, rm, rd, st.row_ptr, st.col_idx, st.col_ptr,
                                                     st.row_idx, wl.scale, dQ, dK, dV, stream), max(args.steps, 5))
    # the entry points that build the work lists on every call, same protocol
    ms_per_call = time_part(lambda: step_per_call(*args_dev), max(args.steps, 5))

    # End to end through the C ABI from pinned host buffers.  Every step copies
    # its inputs host -> device and its outputs (O, statistics, dQ, dK, dV)
    # device -> host inside the timed region; the copies of neighbouring steps
    # overlap the kernels on two copy streams (inputs and outputs
    # double-buffered on the device), as a training loop feeding the GPU would.
    # No L2 flush here: each step's inputs arrive fresh from the host.
    pin = [t.pin_memory() for t in (hQ, hK, hV, hdO)]
    outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (O, rm, rd, dQ, dK, dV)]
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    bufs = [args_dev, tuple(torch.empty_like(t) for t in args_dev)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(args.steps)]
    ev_done = [torch.cuda.Event() for _ in range(args.steps)]
    ev_out = [torch.cuda.Event() for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(world)
    t0.record(s_in)
    for i in range(args.steps):
        b = bufs[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_done[i - 2])  # the buffer's previous step has read its inputs
            for d_, h_ in zip(b[:4], pin):
                d_.copy_(h_, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])  # the buffer's previous outputs are on the host
        step(*b)
        ev_done[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[i])
            for h_, d_ in zip(outs_h, b[4:]):
                h_.copy_(d_, non_blocking=True)
            ev_out[i].record(s_out)
    s_out.wait_stream(s_in)
    t1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), world) / args.steps
    bsr.bsr_attn_check()
    del bufs

    flops = alg_flops(wl, nnzb)
    value = world * flops / (ms_per_step * 1e-3) / 1e12
    peaks = load_peaks()
    kern = {k: {"launches": n, "ms_per_launch": ms / max(n, 1)} for k, (n, ms) in prof.items()}
    for k, rec in kern.items():  # each kernel against its own roof
        kb, kf = kernel_bytes(k, wl, nnzb), kernel_flops(k, wl, nnzb)
        if kb and rec["ms_per_launch"] > 0:
            rec["hbm_frac"] = round(kb / (rec["ms_per_launch"] * 1e-3) / 1e9 / peaks["hbm"], 4)
        elif kf and rec["ms_per_launch"] > 0:
            rec["tensor_frac"] = round(kf / (rec["ms_per_launch"] * 1e-3) / 1e12 / peaks["bf16"], 4)
    dom = max(prof.items(), key=lambda kv: kv[1][1]) if prof else None
    roofline = None
    if dom and kernel_bytes(dom[0], wl, nnzb):
        name, (n, ms) = dom
        kb = kernel_bytes(name, wl, nnzb)
        avg_ms = ms / n
        achieved = kb / (avg_ms * 1e-3) / 1e9
        roofline = {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm"], "traffic": measured_traffic(wl.name, name),
                    "traffic_unit": "bytes per launch (ncu DRAM)", "peak_source": peaks["source"] + " HBM copy",
                    "bytes_per_launch": kb, "ms_per_launch": avg_ms}
    elif dom:
        name, (n, ms) = dom
        kf = kernel_flops(name, wl, nnzb)
        avg_ms = ms / n
        achieved = kf / (avg_ms * 1e-3) / 1e12 if kf else None
        roofline = {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16"],
                    "unit": "TFLOP/s", "frac": (achieved / peaks["bf16"]) if achieved else None,
                    "traffic": measured_traffic(wl.name, name), "traffic_unit": "bytes per launch (ncu DRAM)",
                    "peak_source": peaks["source"] + " bf16 burst"
                    + (" (fp16 operands: the same dense rate as bf16 nominally)" if wl.dtype == "f16" else ""),
                    "flop_per_launch": kf, "ms_per_launch": avg_ms}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "statistic": "median of the per-step times",
        "ms_per_step_mean": round(ms_mean, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": workload_config(wl, nnzb, world, args.forward),
        "ms_fwd": round(ms_fwd, 4), "ms_bwd": round(ms_bwd, 4),
        "api": "bsr_attn_fwd_plan + bsr_attn_bwd_plan on one plan built before timing" if planned
               else "bsr_attn_fwd + bsr_attn_bwd (work lists built on every call)",
        "per_call_api_ms_per_step": round(ms_per_call, 4),
        "kernel_timing": {"pass": "second pass of the same K steps with CUDA events around every launch "
                                  "(on a plan the dK/dV walk and then the dQ walk over its stored dS tiles run "
                                  "in sequence in both passes; per call the recomputing dQ walk overlaps dK/dV "
                                  "on two streams, one after the other in this pass)",
                          "ms_per_step": round(ms_per_step_instr, 4)},
        "pct_of_bf16_peak": round(100 * value / world / peaks["bf16"], 2),
        "long_run": {"steps": long_steps, "ms_per_step_median": round(ms_long, 4),
                     "ms_per_step_mean": round(ms_long_mean, 4),
                     "tflops_median": round(world * flops / (ms_long * 1e-3) / 1e12, 3)},
        "alg_gflop_per_step": flops / 1e9,
        "kernels": kern,
        "gpu_launches": sum(n for n, _ in prof.values()),
        "roofline": roofline,
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "inputs copied in and outputs copied out every step on two copy streams, "
                            "overlapping the neighbouring steps' kernels (double-buffered on the device)"},
        "clocks": clk.summary(),
    }
    if args.sdpa:
        line["sdpa"] = sdpa_comparators(Q, K, V, dO, bm, l2, stream, dev, args)
    if args.other_workloads and world == 1:
        del Q, K, V, dO, O, rm, rd, dQ, dK, dV, args_dev
        line["other_workloads"] = other_workloads(wl.name, dev, args, l2, stream, peaks)
    return line


OTHER_WORKLOADS = ("tiny", "dilated_s2048", "global_s8192_f32", "local_s8192_d256", "local_s8192_d512",
                   "random_p0.01", "random_p0.05", "random_p0.13", "random_p0.27", "random_p0.5")


def other_workloads(headline, dev, args, l2, stream, peaks):
    """fwd+bwd of every other configuration the metric names, same protocol (L2 flushed before every step,
    CUDA events on the stream, median of `args.steps` steps after `args.warmup`): ms, TFLOP/s over stored
    blocks and fraction of the bf16 peak; the density sweep also times dense masked SDPA on the same inputs."""
    import block_sparse_attention_bsr_gb300 as bsr

    out = {}
    for name in OTHER_WORKLOADS:
        if name == headline:
            continue
        wl = inputs.WORKLOADS[name]
        bm = wl.block_mask()
        rp, ci = inputs.bsr_from_block_mask(bm)
        st = bsr.Structure(rp, ci, wl.nb, dev)
        Q, K, V, dO = (t.to(dev) for t in wl.inputs(seed=0))
        O = torch.empty_like(Q)
        rm = torch.empty(Q.shape[:3], device=dev, dtype=torch.float32)
        rd = torch.empty_like(rm)
        dQ, dK, dV = (torch.empty_like(Q) for _ in range(3))

        plan = st.plan(Q)

        def step():
            bsr.bsr_attn_fwd_plan(plan, Q, K, V, wl.scale, O, rm, rd, stream)
            bsr.bsr_attn_bwd_plan(plan, Q, K, V, O, dO, rm, rd, wl.scale, dQ, dK, dV, stream)

        ms = median_call_ms(step, args, l2, stream, dev)
        bsr.profile_collect()
        bsr.profile_enable(True)
        step()
        torch.cuda.synchronize(dev)
        bsr.profile_enable(False)
        kern = {k: round(t * 1e3 / n, 2) for k, (n, t) in bsr.profile_collect().items()}
        bsr.bsr_attn_check()
        flops = alg_flops(wl, st.nnzb)
        tf = flops / (ms * 1e-3) / 1e12
        e = {"ms": round(ms, 4), "tflops": round(tf, 3), "frac_of_bf16_peak": round(tf / peaks["bf16"], 4),
             "dtype": wl.dtype, "shape": [wl.batch, wl.heads, wl.seq, wl.head_dim], "mask": wl.mask,
             "nnzb": st.nnzb, "density": round(st.nnzb / wl.nb ** 2, 4), "kernel_us_one_step": kern}
        if name.startswith("random_p") and args.sdpa:
            e["sdpa_masked_fwd_bwd_ms"] = sdpa_comparators(Q, K, V, dO, bm, l2, stream, dev, args,
                                                           kinds=("masked",))["sdpa_masked_fwd_bwd_ms"]
        out[name] = e
        del Q, K, V, dO, O, rm, rd, dQ, dK, dV, plan, st
        torch.cuda.empty_cache()
    return out


def workload_config(wl, nnzb, world, forward):
    return {"workload": wl.name, "batch": wl.batch, "heads": wl.heads, "seq": wl.seq, "head_dim": wl.head_dim,
            "block": BLOCK, "mask": wl.mask, "radius": wl.radius, "nnzb": nnzb,
            "density": round(nnzb / wl.nb ** 2, 4), "l2": "flushed before every step",
            "parallelism": f"replicas x{world}", "forward": forward}


def sdpa_comparators(Q, K, V, dO, bm, l2, stream, dev, args, kinds=("masked", "dense")):
    """Dense masked SDPA (boolean element mask) and unmasked dense SDPA on the same GPU, fwd+bwd ms."""
    F = torch.nn.functional
    em = torch.from_numpy(np.repeat(np.repeat(bm, BLOCK, 0), BLOCK, 1)).to(dev)
    res = {}
    for name, mask in (("masked", em), ("dense", None)):
        if name not in kinds:
            continue
        def fb():
            q, k, v = (t.detach().requires_grad_() for t in (Q, K, V))
            o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask)
            o.backward(dO)
        try:
            for _ in range(2):
                fb()
            ts = []
            for _ in range(5):
                flush_l2(l2)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fb()
                b.record()
                torch.cuda.synchronize(dev)
                ts.append(a.elapsed_time(b))
            res[f"sdpa_{name}_fwd_bwd_ms"] = round(statistics.median(ts), 4)
        except Exception as e:  # report and continue
            res[f"sdpa_{name}_fwd_bwd_ms"] = f"failed: {type(e).__name__}: {str(e)[:100]}"
    return res


def cpu_baseline(wl, budget_s):
    """The fp64 oracle on the host cores over a bounded sample: whole heads of the workload, fwd+bwd."""
    import oracle

    bm = wl.block_mask()
    nnzb = int(bm.sum())
    hQ, hK, hV, hdO = wl.inputs(seed=0)
    heads, t0 = 0, time.perf_counter()
    while True:
        b, h = divmod(heads, wl.heads)
        b %= wl.batch
        oracle.attn_fwd_bwd_head(hQ[b, h].double().numpy(), hK[b, h].double().numpy(), hV[b, h].double().numpy(),
                                 hdO[b, h].double().numpy(), bm, wl.scale)
        heads += 1
        el = time.perf_counter() - t0
        if el >= budget_s or heads >= wl.batch * wl.heads:
            break
    flops = 14 * BLOCK * BLOCK * wl.head_dim * nnzb * heads
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{heads} of {wl.batch * wl.heads} (batch, head) slices of {wl.name}, fwd+bwd, "
                      f"dense fp64 numpy, {el:.1f} s", "seconds": el, "heads": heads}


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    # NCCL reduces device tensors; other backends (gloo) host tensors
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


SPMM_DENSITIES = (0.01, 0.05, 0.13, 0.27, 0.5, 1.0)


def median_call_ms(fn, args, l2, stream, dev):
    """Median ms of `fn` over args.steps calls after args.warmup, L2 flushed before each, CUDA events on `stream`."""
    for _ in range(args.warmup):
        flush_l2(l2)
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        flush_l2(l2)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize(dev)
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def one_call_kernels(fn, dev):
    """{kernel: us} of one call with per-launch timing on."""
    import block_sparse_attention_bsr_gb300 as bsr

    bsr.profile_collect()
    bsr.profile_enable(True)
    fn()
    torch.cuda.synchronize(dev)
    bsr.profile_enable(False)
    return {k: round(t * 1e3 / n, 2) for k, (n, t) in bsr.profile_collect().items()}


def run_spmm_sweep(args, dev):
    """bsr_spmm on an 8192 x 8192 BSR matrix (64 x 64 blocks of 128) times 8192 x width, bf16, one JSON
    line per block density, beside dense torch.matmul of the same operands on the same GPU."""
    import block_sparse_attention_bsr_gb300 as bsr

    l2 = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        return median_call_ms(fn, args, l2, stream, dev)

    cases = [(p, None) for p in SPMM_DENSITIES] + [(0.05, "rows 0-3 full")]
    for p, skew in cases:
        bm, blocks, X = inputs.make_spmm(64, 64, args.width, p, "bf16", seed=0)
        if skew:  # a few dense block rows among sparse ones: the longest row bounds a one-CTA-per-row walk
            g = torch.Generator().manual_seed(7)
            bm[:4, :] = True
            blocks = torch.randn(int(bm.sum()), BLOCK, BLOCK, generator=g).to(torch.bfloat16)
        rp, ci = inputs.bsr_from_block_mask(bm)
        nnzb = int(bm.sum())
        blocks_d, X_d = blocks.to(dev), X.to(dev)
        rp_d, ci_d = torch.from_numpy(rp).to(dev), torch.from_numpy(ci).to(dev)
        Y = torch.empty(64 * BLOCK, args.width, dtype=torch.bfloat16, device=dev)
        # the dense operand of the comparison: A with zeros outside the stored blocks
        A = torch.zeros(64 * BLOCK, 64 * BLOCK, dtype=torch.bfloat16, device=dev)
        rows = np.repeat(np.arange(64), np.diff(rp))
        for j, (m, k) in enumerate(zip(rows, ci)):
            A[m * BLOCK:(m + 1) * BLOCK, k * BLOCK:(k + 1) * BLOCK] = blocks_d[j]
        ms = timed(lambda: bsr.bsr_spmm(blocks_d, rp_d, ci_d, 64, 64, X_d, Y, stream))
        bsr.bsr_attn_check()
        kern = one_call_kernels(lambda: bsr.bsr_spmm(blocks_d, rp_d, ci_d, 64, 64, X_d, Y, stream), dev)
        dense_ms = timed(lambda: torch.matmul(A, X_d))
        flops = 2 * BLOCK * BLOCK * args.width * nnzb
        print(json.dumps({"op": "bsr_spmm", "metric": "ms per Y = A X, 8192 x 8192 BSR (blocks of 128) x 8192 x width",
                          "density": round(nnzb / 64 ** 2, 4), "nnzb": nnzb, "structure": skew or "iid blocks", "width": args.width, "dtype": "bf16",
                          "ms": round(ms, 4), "dense_matmul_ms": round(dense_ms, 4),
                          "speedup_vs_dense": round(dense_ms / ms, 3),
                          "tflops_over_stored_blocks": round(flops / (ms * 1e-3) / 1e12, 2),
                          "kernel_us_one_call": kern,
                          "steps": args.steps, "warmup": args.warmup, "l2": "flushed before every call",
                          "data": "synthetic"}), flush=True)


SCREEN_THRESHOLDS = (1e-6, 1e-4, 1e-2, 1e-1)


def run_screen_sweep(args, dev):
    """bsr_screened_spmm at n = 8192 (bounds decaying along the diagonal) times 8192 x width, bf16, one
    JSON line per threshold, beside the unfused dense (A * mask) @ B and the plain A @ B on the same GPU."""
    import block_sparse_attention_bsr_gb300 as bsr

    n = 8192
    l2 = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        return median_call_ms(fn, args, l2, stream, dev)

    hA, hdiag, hB = inputs.make_screened(n, args.width, "bf16", seed=0)
    A, diag, B = hA.to(dev), hdiag.to(dev), hB.to(dev)
    C = torch.empty(n, args.width, dtype=torch.bfloat16, device=dev)
    q = diag.abs().sqrt()
    for thr in SCREEN_THRESHOLDS:
        mask = (q[:, None] * q[None, :]) > torch.tensor(thr, dtype=torch.float32, device=dev).sqrt()
        kept = float(mask.float().mean())
        maskb = mask.to(torch.bfloat16)
        ms = timed(lambda: bsr.bsr_screened_spmm(A, diag, B, thr, C, stream))
        bsr.bsr_attn_check()
        kern = one_call_kernels(lambda: bsr.bsr_screened_spmm(A, diag, B, thr, C, stream), dev)
        unfused_ms = timed(lambda: torch.matmul(A * maskb, B))
        dense_ms = timed(lambda: torch.matmul(A, B))
        print(json.dumps({"op": "bsr_screened_spmm", "metric": "ms per C = (A o M) B, n = 8192, B 8192 x width",
                          "threshold": thr, "kept_fraction": round(kept, 4), "width": args.width, "dtype": "bf16",
                          "ms": round(ms, 4), "unfused_masked_matmul_ms": round(unfused_ms, 4),
                          "dense_matmul_ms": round(dense_ms, 4),
                          "speedup_vs_unfused": round(unfused_ms / ms, 3), "kernel_us_one_call": kern,
                          "steps": args.steps,
                          "warmup": args.warmup, "l2": "flushed before every call", "data": "synthetic"}),
              flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="global_s8192", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--forward", default="online", choices=["online", "two-pass"],
                    help="forward variant: the online-softmax pass, or the statistics-first two-pass variant")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--api", default="plan", choices=["plan", "per-call"],
                    help="entry points of the step: a reusable plan built once, or the per-call ones")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the oracle CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sdpa", action=argparse.BooleanOptionalAction, default=True,
                    help="also time dense masked / unmasked SDPA on the same GPU")
    ap.add_argument("--other-workloads", action=argparse.BooleanOptionalAction, default=True,
                    help="also time every other configuration (tiny, dilated, fp32, head_dim 256 / 512, densities)")
    ap.add_argument("--spmm-sweep", action="store_true",
                    help="instead of attention: bsr_spmm against dense matmul over block densities (one line each)")
    ap.add_argument("--screen-sweep", action="store_true",
                    help="instead of attention: bsr_screened_spmm against the unfused masked matmul over thresholds")
    ap.add_argument("--width", type=int, default=512, help="columns of X / B for --spmm-sweep / --screen-sweep")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    wl = inputs.WORKLOADS[args.workload]
    if args.spmm_sweep or args.screen_sweep:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        (run_spmm_sweep if args.spmm_sweep else run_screen_sweep)(args, dev)
        return

    if args.impl == "reference":
        # The CPU oracle stands as the reference arm; rank 0 alone runs it.  A
        # whole step (all B * H slices of seq 8192, ~1.5 s of fp64 each) would
        # not fit a few minutes, so one reference step is ONE (batch, head)
        # slice of the workload, fwd+bwd, and value / ms_per_step are for that
        # slice; the full-step time is reported separately, extrapolated.
        if rank != 0:
            return
        import oracle

        bm = wl.block_mask()
        nnzb = int(bm.sum())
        hQ, hK, hV, hdO = wl.inputs(seed=0)
        times = []
        for i in range(args.warmup + args.steps):
            b, h = divmod(i % (wl.batch * wl.heads), wl.heads)
            t0 = time.perf_counter()
            oracle.attn_fwd_bwd_head(*(t[b, h].double().numpy() for t in (hQ, hK, hV, hdO)), bm, wl.scale)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        sec = statistics.median(times)
        flops_head = 14 * BLOCK * BLOCK * wl.head_dim * nnzb
        v = flops_head / sec / 1e12
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        sample = (f"one (batch, head) slice of {wl.name} per step ({wl.batch * wl.heads} slices make a full step), "
                  f"fwd+bwd, dense fp64 numpy, median {sec:.2f} s")
        line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
                "step": "one (batch, head) slice of the workload",
                "ms_per_full_step_extrapolated": round(sec * 1e3 * wl.batch * wl.heads, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_config(wl, nnzb, 1, args.forward),
                "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    # CPU oracle baseline first, on rank 0 at N=1, before any GPU work
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    if world > 1:
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
        dev = torch.device("cuda", local)
    else:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
    line = run_ours(args, rank, world, dev)
    if cpu is not None:
        line["cpu_baseline"] = {k: (round(v, 6) if isinstance(v, float) else v) for k, v in cpu.items()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
