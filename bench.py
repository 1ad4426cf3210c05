#!/usr/bin/env python
"""Benchmark of the GB300 ragged-M grouped GEMM (one JSON line per run).

A step is one launch of the whole hot path: Y_e = X_e . W_e for every expert
of one batch of synthetic input (offsets -> tile list -> TMA -> tcgen05 ->
epilogue, all inside the kernel).  The metric is useful TFLOP/s,
2 * M_tot * K * N / t ("Grouped GEMM for Imbalanced Experts on Blackwell: A WIP
Worklog", section 1), with t measured on the device with CUDA events around K
replays of one step captured in a CUDA graph (the same K steps launched one by
one from the host are reported beside it as "eager").

Headline workload (the default): prefill-scale routing, the largest of the
workloads -- 32 experts, K = 6144, N = 4096, 32 768 tokens each routed to one
uniformly random expert.  Beside it, in the same JSON line ("configs"), the
other workloads are timed in the same way: the worklog's uniform and skewed
16k-row routings (section 1, "Some Results First") and the skewed one at 2k
rows, the small-decode shape (32 experts x 16 rows, the decode example of
"Pearl's grouped GEMM kernel for MoE models, explained", "Why MoE needs a
grouped GEMM"), and the skewed routings once more with the tile shape planned
from the device offsets alone.  Every workload's inputs are larger than the
129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
experts of one GPU under expert parallelism, no data-path collective: weak
scaling); rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from ragged_grouped_gemm_02_gb300 import workloads as wl  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "ragged_grouped_gemm_02_gb300", "csrc")
L2_BYTES = 129 * 1024 * 1024
METRIC = "useful TFLOP/s (2*M_tot*K*N/t) and HBM GB/s, as % of GB300 roofline"
# The worklog's own figure for this exact metric and workload (B300, k2 with
# two stages, uniform routing 16k rows): context, another machine's number.
PAGE_NUMBERS = {"uniform": 440.1}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default="prefill", choices=sorted(wl.WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="time only the headline workload (no uniform / skew / decode side configurations)")
    p.add_argument("--bm", type=int, default=0)
    p.add_argument("--bn", type=int, default=0)
    p.add_argument("--stages", type=int, default=0)
    p.add_argument("--tail64", type=int, default=0, help="0 auto, 1 on, -1 off")
    p.add_argument("--gather-mode", type=int, default=0, help="gather ops: 0 auto, 1 TMA gather4, 2 two-pass")
    p.add_argument("--mixed", type=int, default=0,
                   help="plain GEMM and fused gate-up: 0 auto, 1 the mixed launch (large experts on CTA pairs "
                        "beside small ones on single CTAs, tiles claimed on the device), 2 the same with fixed "
                        "walks, -1 off")
    p.add_argument("--mixed-pair-sms", type=int, default=0,
                   help="mixed launch: SMs of the pair kernel (0: split by estimated work, -1: none)")
    p.add_argument("--walk-order", type=int, default=0,
                   help="0 auto, -1 list order, 1 front/back interleave, 2 scatter, 3 size-sorted interleave, "
                        "4 N-major within each expert")
    p.add_argument("--op", default="gemm", choices=["gemm", "swiglu", "fp8", "gather", "swiglu_gather"],
                   help="gemm: Y = X.W; swiglu: the workload's weights read as [gate | up], "
                        "H = silu(X.W_gate) * (X.W_up) with N/2 output columns; fp8: the same draws "
                        "quantised to E4M3 with per-row / per-column scales; gather / swiglu_gather: "
                        "the activations held as M_tot tokens in token order, each routed row read "
                        "through its token index inside the kernel")
    p.add_argument("--profile", action="store_true",
                   help="for ncu: --warmup launches then one more, no timing, no CPU work after")
    p.add_argument("--no-host-counts", action="store_true",
                   help="with --profile: plan from the device offsets alone (no host counts)")
    return p.parse_args()


# ------------------------------------------------------------------ helpers

def dist_setup(backend):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash():
    h = hashlib.sha256()
    for path in sorted(glob.glob(os.path.join(CSRC, "*"))):
        if path.endswith((".cu", ".cuh", ".h")):
            h.update(os.path.basename(path).encode())
            with open(path, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources and this workload; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("kernel_hash") != kernel_source_hash():
        return None
    entry = t.get("workloads", {}).get(workload)
    return None if entry is None else int(entry["bytes_per_launch"])


def work_of(counts, K, N):
    M = int(np.sum(counts))
    active = int(np.count_nonzero(counts))
    flops = 2.0 * M * K * N
    # each active expert's weights once, X and Y once, the offsets
    bytes_ = 2.0 * (active * K * N + M * K + M * N) + 4.0 * (len(counts) + 1)
    return flops, bytes_


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="rgg_clocks_", suffix=".csv")
        os.close(fd)
        try:
            phys = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
            idx = phys[self.dev] if self.dev < len(phys) and phys[self.dev] != "" else str(self.dev)
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", idx], stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def oracle_cpu_rate(inp, budget_s=12.0, op="gemm", scales=None, row_index=None):
    """The fp64 oracle as it stands, on the host cores, over a bounded sample
    of the workload: the first experts' complete rows (all N columns), about
    `budget_s` of work.  Returns (TFLOP/s, sample description, threads)."""
    import oracle
    oracle.build()
    counts = inp.counts
    K, N = inp.X.shape[1], inp.W.shape[2]
    threads = oracle.max_threads()
    if op == "fp8":
        xb, wb = wl.fp8_codes(inp.X), wl.fp8_codes(inp.W)
        sxn, swn = scales[0].numpy(), scales[1].numpy()

        def fn(x, w, off, r0=0, e0=0):
            return oracle.grouped_gemm_fp8(x, w, sxn[r0:r0 + x.shape[0]], swn[e0:e0 + w.shape[0]], off)
    elif row_index is not None:
        # the gathered ops: the oracle's gather of the sample's rows, then its product
        xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
        base = oracle.grouped_swiglu if op == "swiglu_gather" else oracle.grouped_gemm

        def fn(x, w, off, r0=0, e0=0):
            return base(oracle.gather_rows(xb, row_index[r0:r0 + x.shape[0]]), w, off)
    else:
        xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
        base = oracle.grouped_swiglu if op == "swiglu" else oracle.grouped_gemm

        def fn(x, w, off, r0=0, e0=0):
            return base(x, w, off)
    # calibrate on one expert's rows (or 16 rows)
    e0 = int(np.argmax(counts > 0))
    r = int(min(counts[e0], 16))
    r0 = int(inp.offsets[e0])
    t0 = time.perf_counter()
    fn(np.ascontiguousarray(xb[r0:r0 + r]), np.ascontiguousarray(wb[e0:e0 + 1]), [0, r], r0, e0)
    rate = 2.0 * r * K * N / max(time.perf_counter() - t0, 1e-6)
    want = budget_s * rate
    e_take, flops = 0, 0.0
    while e_take < len(counts) and (flops < want or flops == 0.0):
        flops += 2.0 * counts[e_take] * K * N
        e_take += 1
    rows = int(inp.offsets[e_take])
    off = inp.offsets[:e_take + 1]
    t0 = time.perf_counter()
    fn(np.ascontiguousarray(xb[:rows]), np.ascontiguousarray(wb[:e_take]), off)
    dt = time.perf_counter() - t0
    sample = "experts 0..%d of %d (%d of %d rows, all %d columns), %.1f GFLOP in %.2f s" % (
        e_take - 1, len(counts), rows, int(counts.sum()), N, flops / 1e9, dt)
    return flops / dt / 1e12, sample, threads


# --------------------------------------------------------------- our arm

def run_profile(args):
    """A short, fixed launch sequence for ncu captures: `--warmup` launches,
    then one more (capture it with -s <warmup> -c 1)."""
    import ragged_grouped_gemm_02_gb300 as rgg
    from ragged_grouped_gemm_02_gb300 import _build
    _build.build()
    dev = torch.device("cuda", 0)
    inp = wl.make_inputs(args.workload)
    X, W = inp.X.to(dev), inp.W.to(dev)
    off = torch.from_numpy(inp.offsets).to(dev)
    Y = torch.empty(X.shape[0], W.shape[2], dtype=torch.bfloat16, device=dev)
    opts = dict(bm=args.bm, bn=args.bn, stages=args.stages, tail64=args.tail64,
                walk_order=args.walk_order, host_counts=None if args.no_host_counts else inp.counts)
    if args.op in ("gemm", "swiglu"):
        opts.update(mixed=args.mixed, mixed_pair_sms=args.mixed_pair_sms)
    if args.op == "gather":
        # the same recipe as the timed gather op: M_tot tokens, distinct tokens per expert
        gen = torch.Generator().manual_seed(inp.workload.seed + 7)
        idx = torch.from_numpy(wl.routed_row_index(inp.counts, X.shape[0], gen)).to(dev)
        opts["gather_mode"] = args.gather_mode
        opts["workspace"] = torch.empty_like(X)  # the two-pass mode's gathered rows

        def launch():
            rgg.rgg_grouped_gemm_gather(X, idx, W, off, Y, **opts)
    elif args.op == "gemm":
        def launch():
            rgg.rgg_grouped_gemm(X, W, off, Y, **opts)
    elif args.op == "swiglu":
        H = torch.empty(X.shape[0], W.shape[2] // 2, dtype=torch.bfloat16, device=dev)

        def launch():
            rgg.rgg_grouped_gemm_swiglu(X, W, off, H, **opts)
    elif args.op == "fp8":
        X8, W8, sx, sw = wl.quantize_fp8(inp.X, inp.W)
        X8, W8, sx, sw = X8.to(dev), W8.to(dev), sx.to(dev), sw.to(dev)
        del X, W

        def launch():
            rgg.rgg_grouped_gemm_fp8(X8, W8, sx, sw, off, Y, **opts)
    else:
        raise SystemExit("--profile covers --op gemm, gather, swiglu and fp8")
    for _ in range(args.warmup + 1):
        launch()
    torch.cuda.synchronize(dev)
    status = rgg.rgg_query_status(0)
    n_plan = inp.workload.N // 2 if args.op == "swiglu" else inp.workload.N
    plan = rgg.rgg_plan(inp.workload.E, inp.X.shape[0], inp.workload.K, n_plan, op=args.op, **opts)
    print(json.dumps({"profile": args.workload, "launches": args.warmup + 1, "status": status, "plan": plan}))
    if status != rgg.RGG_OK:
        raise SystemExit(1)


class Step:
    """One workload and op on the device: inputs resident in HBM, the launch
    of one step, its algorithmic work and what the end-to-end run copies."""

    def __init__(self, rgg, args, workload, op, rank, dev, host_counts=True):
        w = wl.WORKLOADS[workload]
        self.rgg, self.op, self.workload, self.dev = rgg, op, workload, dev
        inp = wl.make_inputs(wl.Workload(**{**w.__dict__, "seed": w.seed + 1000 * rank}))
        self.w, self.inp = w, inp
        K, N, E = w.K, w.N, w.E
        self.K, self.N, self.E = K, N, E
        M_tot = inp.X.shape[0]
        self.M_tot = M_tot
        flops, bytes_ = work_of(inp.counts, K, N)
        self.fused = op in ("swiglu", "swiglu_gather")
        self.gather = op in ("gather", "swiglu_gather")
        self.N_out = N // 2 if self.fused else N
        if self.fused:  # the output is half as wide; the weight bytes and MMA work are the same
            bytes_ -= 2.0 * M_tot * (N - self.N_out)
        self.sx = self.sw = self.idx_h = None
        gemm = rgg.rgg_grouped_gemm_swiglu if self.fused else rgg.rgg_grouped_gemm
        if op == "fp8":
            # the same draws quantised to E4M3 with per-row / per-column scales:
            # X and W stream at one byte per element, scales are fp32
            X8, W8, sx, sw = wl.quantize_fp8(inp.X, inp.W)
            active = int(np.count_nonzero(inp.counts))
            bytes_ = (1.0 * (active * K * N + M_tot * K) + 2.0 * M_tot * N + 4.0 * (M_tot + E * N)
                      + 4.0 * (E + 1))
            self.sx, self.sw = sx, sw
            self.sx_d, self.sw_d = sx.to(dev), sw.to(dev)
            inp.X, inp.W = X8, W8

            def gemm(Xd, Wd, offd, Yd, sxd=None, **kw):
                return rgg.rgg_grouped_gemm_fp8(Xd, Wd, self.sx_d if sxd is None else sxd, self.sw_d, offd, Yd, **kw)
        if self.gather:
            # The activations are M_tot tokens in token order; routed row i reads
            # token row_index[i] (each expert's rows are distinct tokens in
            # increasing order).  The index adds 4 bytes per routed row.
            gen = torch.Generator().manual_seed(w.seed + 1000 * rank + 7)
            self.idx_h = torch.from_numpy(wl.routed_row_index(inp.counts, M_tot, gen))
            self.idx_d = self.idx_h.to(dev)
            bytes_ += 4.0 * M_tot
            gfn = rgg.rgg_grouped_gemm_swiglu_gather if self.fused else rgg.rgg_grouped_gemm_gather

            def gemm(Xd, Wd, offd, Yd, idx=None, **kw):
                return gfn(Xd, self.idx_d if idx is None else idx, Wd, offd, Yd, **kw)
        self.gemm = gemm
        self.flops, self.bytes = flops, bytes_
        self.X, self.W = inp.X.to(dev), inp.W.to(dev)
        self.off = torch.from_numpy(inp.offsets).to(dev)
        self.Y = torch.empty(M_tot, self.N_out, dtype=torch.bfloat16, device=dev)
        # The tile shape is planned from the routed counts, known on the host as
        # in the worklog's harness (host_counts=False: from the device offsets
        # alone); the kernel itself reads the offsets on the device.
        self.opts = dict(bm=args.bm, bn=args.bn, stages=args.stages, tail64=args.tail64,
                         walk_order=args.walk_order, host_counts=inp.counts if host_counts else None)
        if op in ("gemm", "swiglu"):
            self.opts.update(mixed=args.mixed, mixed_pair_sms=args.mixed_pair_sms)
        self.plan_from = ("host-side routed counts (tile shape only)" if host_counts
                          else "device offsets only (no host counts)")
        # the key of this launch's DRAM capture in profiles/dram_traffic.json
        self.traffic_key = (workload if op == "gemm" else workload + "+" + op) + ("" if host_counts
                                                                                 else " (device offsets)")
        if self.gather:
            self.opts["gather_mode"] = args.gather_mode
            # the two-pass mode's gathered rows, allocated once outside the timed region
            self.opts["workspace"] = torch.empty_like(self.X)
        self.plan = rgg.rgg_plan(E, M_tot, K, self.N_out,
                                 num_sms=torch.cuda.get_device_properties(dev).multi_processor_count,
                                 op=op, **self.opts)
        # launches of this library's kernels in one step: the two-pass gather runs
        # its row gather and then the grouped GEMM, the mixed launch its pair
        # kernel and its 1-CTA kernel (each when it has SMs), every other op one kernel
        if self.plan.get("mixed"):
            self.per_step = int(self.plan["grid"] > 0) + int(self.plan["single_grid"] > 0)
        else:
            self.per_step = 2 if self.plan.get("gather_mode") == 2 else 1

    def launch(self, stream):
        self.gemm(self.X, self.W, self.off, self.Y, stream=stream, **self.opts)


def time_step(step, args, world, dev, ramp_s):
    """W warm-up steps (after an untimed ramp of about `ramp_s` seconds that
    brings the GPU to its clocks under load), then K steps launched one by one
    (eager) and K replays of one step captured in a CUDA graph (the timed
    region), on the launching stream, bracketed by a barrier and a device
    synchronisation.  Returns the timings and the clock record."""
    rgg = step.rgg
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev.index)
    sampler.start()
    t_begin = time.time()
    ramp = 0
    while time.time() - t_begin < ramp_s:
        step.launch(stream)
        ramp += 1
        if ramp % 64 == 0:
            torch.cuda.synchronize(dev)
    for _ in range(max(3, args.warmup)):
        step.launch(stream)
    status = rgg.rgg_query_status(dev.index, stream)
    if status != rgg.RGG_OK:
        raise RuntimeError("device status after warm-up: %s" % rgg.rgg_status_string(status))
    K_steps = args.steps

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    start.record(stream)
    for _ in range(K_steps):
        step.launch(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    status = rgg.rgg_query_status(dev.index, stream)
    if status != rgg.RGG_OK:
        raise RuntimeError("device status after the eager steps: %s" % rgg.rgg_status_string(status))
    eager_ms = max_over_ranks(start.elapsed_time(end), world, dev)

    # Timed region: the K steps captured back to back in one CUDA graph and
    # replayed once on the same stream, so the device time has no host launch
    # work in it (the pages time their kernels inside CUDA graphs too).  Each
    # step's kernels are launched with programmatic stream serialisation, so a
    # step's CTAs become resident as the previous step's CTAs leave and wait
    # on the device for it, as in a model's forward graph.  For comparison,
    # the same K steps as K replays of a one-step graph (each replay pays the
    # graph launch) are timed after it and reported beside it.
    timing = "cuda_graph: the K steps captured in one graph, replayed once"
    graph_replay_ms = None
    try:
        gk = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gk):
            for _ in range(K_steps):
                step.launch(torch.cuda.current_stream(dev))
        gk.replay()
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        g0.record(stream)
        gk.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        total_ms = max_over_ranks(g0.elapsed_time(g1), world, dev)
        del gk
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step.launch(torch.cuda.current_stream(dev))
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(K_steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        graph_replay_ms = max_over_ranks(g0.elapsed_time(g1), world, dev)
        del g
    except RuntimeError as e:
        timing = "eager (graph capture failed: %s)" % str(e)[:160]
        total_ms = eager_ms
    clocks = sampler.stop()
    status = rgg.rgg_query_status(dev.index, stream)
    if status != rgg.RGG_OK:
        raise RuntimeError("device status after the timed region: %s" % rgg.rgg_status_string(status))
    return {"total_ms": total_ms, "eager_ms": eager_ms, "graph_replay_ms": graph_replay_ms, "timing": timing,
            "clocks": clocks,
            "ramp": {"steps": ramp, "seconds": round(ramp_s, 2),
                     "note": "untimed launches before the warm-up, so the clocks are those under load"}}


def graph_replay_of(step, t, K_steps, world):
    """The K steps timed as K replays of a one-step CUDA graph (each replay
    pays the graph launch), beside the timed region's one graph of K steps."""
    if t.get("graph_replay_ms") is None:
        return None
    return {"value": round(step.flops * K_steps * world / (t["graph_replay_ms"] / 1e3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(t["graph_replay_ms"] / K_steps, 5),
            "note": "the same K steps as K replays of a one-step CUDA graph"}


def roofline_of(step, launch_ms, peaks):
    """Achieved algorithmic bytes (or FLOPs) per launch over the launch time,
    against the measured peak of the bound that is larger."""
    op = step.op
    t_hbm = step.bytes / (peaks["hbm_gbs"] * 1e9)
    # a contraction is measured against the peak of its own operand type: FP8
    # takes the measured bf16 peak times the nominal fp8/bf16 ratio (2)
    tc_peak = peaks["bf16_tflops"] * (2.0 if op == "fp8" else 1.0)
    t_tc = step.flops / (tc_peak * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": round(step.bytes / (launch_ms / 1e3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": round(step.flops / (launch_ms / 1e3) / 1e12, 1),
                "peak": tc_peak, "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    # the capture of this exact launch: the workload, and the op when it is not the plain GEMM
    roof["traffic"] = measured_traffic(step.traffic_key)
    roof["peak_source"] = peaks["source"] + (" bf16 x 2 (nominal fp8/bf16 ratio)" if op == "fp8" else "")
    roof["algorithmic_per_launch"] = {"flops": step.flops, "bytes": step.bytes}
    roof["launch_ms"] = round(launch_ms, 5)
    if step.plan.get("mixed"):
        roof["launch_scope"] = ("one step of the CUDA-graph timed region: the mixed launch (its pair kernel and "
                                "its 1-CTA kernel side by side)")
    elif step.per_step == 2:
        roof["launch_scope"] = "one step of the CUDA-graph timed region: the row gather and the GEMM"
    else:
        roof["launch_scope"] = "one GEMM launch in the CUDA-graph timed region"
    roof["hbm_gbs"] = round(step.bytes / (launch_ms / 1e3) / 1e9, 1)
    roof["hbm_frac"] = round(step.bytes / (launch_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)
    roof["tensor_frac"] = round(step.flops / (launch_ms / 1e3) / 1e12 / tc_peak, 4)
    # The measured sustained bf16 rate (a seconds-long GEMM loop under the power cap) is the
    # fairer yardstick for shapes that draw the cap during a long back-to-back loop; the
    # burst figure above stays the roofline's denominator.
    tc_sust = peaks["bf16_tflops_sustained"] * (2.0 if op == "fp8" else 1.0)
    roof["tensor_frac_of_sustained"] = round(step.flops / (launch_ms / 1e3) / 1e12 / tc_sust, 4)
    return roof


def e2e_of(step, args, world, dev):
    """The same metric end to end through the public API: every step copies
    its inputs (X, the offsets, and for FP8 the row scales, for the gather ops
    the token indices) in from pinned host memory and its result out to pinned
    host memory, all inside the timed region.  As in a serving loop, two
    buffer sets let step i's copies overlap the GEMM of its neighbours: inputs
    go in on one stream, results come out on another, events keep each buffer
    from being overwritten while it is still in use."""
    rgg = step.rgg
    K_steps = args.steps
    stream = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    inp = step.inp
    hX = inp.X.pin_memory()
    hoff = torch.from_numpy(inp.offsets).pin_memory()
    hY = [torch.empty(step.M_tot, step.N_out, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dX = [torch.empty_like(step.X) for _ in range(2)]
    doff = [torch.empty_like(step.off) for _ in range(2)]
    dY = [step.Y, torch.empty_like(step.Y)]
    fp8, gather = step.op == "fp8", step.gather
    if fp8:
        hsx = step.sx.pin_memory()
        dsx = [torch.empty_like(step.sx_d) for _ in range(2)]
    if gather:
        hidx = step.idx_h.pin_memory()
        didx = [torch.empty_like(step.idx_d) for _ in range(2)]
    opts = step.opts

    def run(b, st):
        if fp8:
            step.gemm(dX[b], step.W, doff[b], dY[b], sxd=dsx[b], stream=st, **opts)
        elif gather:
            step.gemm(dX[b], step.W, doff[b], dY[b], idx=didx[b], stream=st, **opts)
        else:
            step.gemm(dX[b], step.W, doff[b], dY[b], stream=st, **opts)

    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, gemm_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for b in range(2):
        gemm_done[b].record(stream)
        out_done[b].record(stream)

    def e2e_step(i):
        b = i % 2
        s_in.wait_event(gemm_done[b])          # the GEMM two steps back has read dX[b]
        with torch.cuda.stream(s_in):
            dX[b].copy_(hX, non_blocking=True)
            doff[b].copy_(hoff, non_blocking=True)
            if fp8:
                dsx[b].copy_(hsx, non_blocking=True)
            if gather:
                didx[b].copy_(hidx, non_blocking=True)
        in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_done[b])         # dY[b] has been read out
        run(b, stream)
        gemm_done[b].record(stream)
        s_out.wait_event(gemm_done[b])
        with torch.cuda.stream(s_out):
            hY[b].copy_(dY[b], non_blocking=True)
        out_done[b].record(s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    e_start.record(stream)
    s_in.wait_event(e_start)
    for i in range(K_steps):
        e2e_step(i)
    s_out.synchronize()
    e_end.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(world)
    e_ms = max_over_ranks(e_start.elapsed_time(e_end), world, dev)

    # The same steps without overlap: copy in, GEMM, copy out, one after the
    # other on one stream (what a caller that waits for each result sees).
    def serial_step():
        with torch.cuda.stream(stream):
            dX[0].copy_(hX, non_blocking=True)
            doff[0].copy_(hoff, non_blocking=True)
            if fp8:
                dsx[0].copy_(hsx, non_blocking=True)
            if gather:
                didx[0].copy_(hidx, non_blocking=True)
            run(0, stream)
            hY[0].copy_(dY[0], non_blocking=True)

    torch.cuda.synchronize(dev)
    barrier(world)
    s_start, s_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_start.record(stream)
    for _ in range(K_steps):
        serial_step()
    s_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    s_ms = max_over_ranks(s_start.elapsed_time(s_end), world, dev)
    status = rgg.rgg_query_status(dev.index, stream)
    if status != rgg.RGG_OK:
        raise RuntimeError("device status after the end-to-end steps: %s" % rgg.rgg_status_string(status))
    h2d = (hX.numel() * hX.element_size() + hoff.numel() * 4 + (hsx.numel() * 4 if fp8 else 0)
           + (hidx.numel() * 4 if gather else 0))
    return {"value": round(step.flops * K_steps * world / (e_ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(hY[0].numel() * 2),
            "ms_per_step": round(e_ms / K_steps, 4),
            "pipeline": "two buffer sets; step i's host copies overlap neighbouring GEMMs",
            "serial": {"value": round(step.flops * K_steps * world / (s_ms / 1e3) / 1e12, 3),
                       "ms_per_step": round(s_ms / K_steps, 4),
                       "note": "copy in, GEMM, copy out in order on one stream"},
            "weights": "resident in HBM (model parameters); not copied per step"}


def config_of(step, world):
    w = step.w
    cfg = {"workload": step.workload + ("" if step.op == "gemm" else "+" + step.op), "op": step.op,
           "E": step.E, "K": step.K, "N": step.N_out, "weight_columns": step.N, "M_tot": step.M_tot,
           "routing": w.routing, "note": w.note, "accumulate": "fp32", "out": "bf16",
           "l2": "inputs larger than L2 (%.0f MB > 129 MB), no flush" % (step.bytes / 1e6)
           if step.bytes > L2_BYTES else "inputs smaller than L2: back-to-back launches",
           "plan": step.plan, "plan_from": step.plan_from, "parallelism": "expert replicas x%d" % world}
    if step.gather:
        cfg.update({"tokens": step.M_tot, "row_index": "each expert's rows are distinct tokens, in token order"})
    return cfg


# The other workloads timed beside the headline, in the same way: the large
# uniform and skewed routings and the small-decode shape, and the skewed
# routings once more with the tile shape planned from the device offsets alone.
SIDE_CONFIGS = [("uniform", True), ("skew16k", True), ("skew2k", True), ("decode", True),
                ("skew16k", False), ("skew2k", False)]


def run_ours(args):
    import ragged_grouped_gemm_02_gb300 as rgg
    from ragged_grouped_gemm_02_gb300 import _build

    world, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    peaks = load_peaks()

    step = Step(rgg, args, args.workload, args.op, rank, dev)
    t = time_step(step, args, world, dev, ramp_s=1.0)
    K_steps = args.steps
    launch_ms = t["total_ms"] / K_steps
    value = step.flops * K_steps * world / (t["total_ms"] / 1e3) / 1e12
    eager = {"value": round(step.flops * K_steps * world / (t["eager_ms"] / 1e3) / 1e12, 3), "unit": "TFLOP/s",
             "ms_per_step": round(t["eager_ms"] / K_steps, 5),
             "note": "the same K steps launched one by one from the host"}
    replay = graph_replay_of(step, t, K_steps, world)
    roof = roofline_of(step, launch_ms, peaks)
    e2e = None if args.no_e2e else e2e_of(step, args, world, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sample, threads = oracle_cpu_rate(step.inp, op=args.op,
                                             scales=(step.sx, step.sw) if args.op == "fp8" else None,
                                             row_index=step.idx_h.numpy() if step.gather else None)
        cpu = {"value": round(v, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample}
    launches = K_steps * step.per_step
    headline_cfg = config_of(step, world)
    del step
    torch.cuda.empty_cache()

    configs = {}
    if not args.no_configs:
        for name, from_counts in SIDE_CONFIGS:
            if name == args.workload and from_counts:
                continue
            s = Step(rgg, args, name, args.op, rank, dev, host_counts=from_counts)
            ts = time_step(s, args, world, dev, ramp_s=0.5)
            lm = ts["total_ms"] / K_steps
            key = name if from_counts else name + " (plan from device offsets)"
            configs[key] = {
                "value": round(s.flops * K_steps * world / (ts["total_ms"] / 1e3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(lm, 5), "roofline": roofline_of(s, lm, peaks), "timing": ts["timing"],
                "graph_replay": graph_replay_of(s, ts, K_steps, world), "clocks": ts["clocks"],
                "config": config_of(s, world)}
            launches += K_steps * s.per_step
            del s
            torch.cuda.empty_cache()

    page = PAGE_NUMBERS.get(args.workload)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K_steps,
        "warmup": args.warmup, "ms_per_step": round(t["total_ms"] / K_steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": round(value / page, 4) if page and args.op == "gemm" else None,
        "dtype": "e4m3" if args.op == "fp8" else "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/K) weights)",
        "config": headline_cfg,
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "timing": t["timing"], "graph_replay": replay,
        "eager": eager,
        "ramp": t["ramp"], "clocks": t["clocks"], "configs": configs,
        "gpu_launches": launches,
        "gpu_launches_note": "kernels of this library launched in the timed regions behind the values: the "
                             "headline's K steps plus each side configuration's K steps (the graph_replay and "
                             "eager figures beside them launch as many again each)", "impl": "ours",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# --------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle as it stands, on the host cores: each step is a bounded
    sample of the workload (the first rows of expert 0, all N columns), sized
    so the whole run takes about a minute."""
    world, rank, _ = dist_setup("gloo")
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w)
    K, N = w.K, w.N
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    e0 = int(np.argmax(inp.counts > 0))
    r0 = int(inp.offsets[e0])
    # calibrate: one row
    t0 = time.perf_counter()
    oracle.grouped_gemm(np.ascontiguousarray(xb[r0:r0 + 1]), wb[e0:e0 + 1], [0, 1])
    per_row = max(time.perf_counter() - t0, 1e-6)
    budget = 60.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(inp.counts[e0], budget / per_row)))
    sub_x = np.ascontiguousarray(xb[r0:r0 + rows])
    sub_w = np.ascontiguousarray(wb[e0:e0 + 1])
    for _ in range(args.warmup):
        oracle.grouped_gemm(sub_x, sub_w, [0, rows])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.grouped_gemm(sub_x, sub_w, [0, rows])
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * K * N * args.steps
    value = flops / dt / 1e12
    sample = "%d rows of expert %d (all %d columns, K=%d) per step" % (rows, e0, N, K)
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "E": w.E, "K": K, "N": N, "M_tot": int(inp.counts.sum())},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
