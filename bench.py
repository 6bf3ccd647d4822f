"""Benchmark of the single-GPU MoE layer path: preprocess -> dispatch_with_permute
-> grouped SwiGLU MLP -> combine, on seeded synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mid] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is one pass of the whole path over one
batch.  `value` is whole-job tokens/s with inputs resident in HBM (device-timed
with CUDA events on the launching stream); `e2e` is the same metric through the
same C-ABI calls with the inputs copied from pinned host memory and the result
copied back inside the timed region.  With N > 1 (torchrun) every rank runs an
independent replica of the workload on its own GPU (the path has no exchange
step on one GPU), a barrier brackets the timed region, the slowest rank's time
is used, and `value` counts every rank's tokens.

`--impl reference` times the CPU oracle (a deliberately slow fp64 restatement)
on a bounded sample of the same workload on the host cores.
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

import workloads  # noqa: E402

METRIC = "MoE-layer tokens/s; permute/combine HBM GB/s; grouped-GEMM TFLOP/s vs peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129e6


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained") if k in d}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def profiled_traffic(workload: str, kernel_source: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a
    kernel, from an ncu summary under profiles/ -- only while the kernel's source
    file still has the hash recorded with the counters, else None."""
    import glob
    import hashlib
    src = os.path.join(ROOT, kernel_source)
    if not os.path.exists(src):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read()
        for block in text.split("```roofline-traffic")[1:]:
            fields = dict(line.split(":", 1) for line in block.split("```")[0].strip().splitlines() if ":" in line)
            fields = {k.strip(): v.strip() for k, v in fields.items()}
            if (fields.get("kernel_source") == kernel_source and fields.get("source_sha256") == digest
                    and fields.get("workload") == workload):
                return int(fields["traffic_bytes_per_launch"])
    return None


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summarize(self.lines)

    @staticmethod
    def summarize(lines):
        """Median SM clock and power, the highest max clock and the throttle
        reasons seen Active, from nvidia-smi CSV lines of QUERY."""
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            try:
                power.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w": round(statistics.median(power), 1) if power else None}


PRE_ROLL_S = 0.5  # seconds of warm replays between the clock sampler's start and a timed region


def pre_roll_count(step_ms: float, minimum: int) -> int:
    """Warm replays that keep the GPU busy for PRE_ROLL_S after the clock sampler
    starts (its first sample comes 0.1-0.2 s later), so that the samples fall
    under load; at least `minimum`."""
    return max(minimum, int(math.ceil(PRE_ROLL_S * 1e3 / max(step_ms, 0.02))))


# ------------------------------------------------------- multi-rank timing

def max_over_ranks(ms: float, device=None) -> float:
    """The slowest rank's time (all ranks get it); identity on one process."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, steps: int, ms_slowest: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world * steps / (ms_slowest / 1e3)


# ----------------------------------------------------------------- problem

class Problem:
    """Device-resident inputs, outputs and workspaces of one MoE layer."""

    def __init__(self, moe, w: workloads.Workload, seed: int, dev, combine_format: str = "bf16",
                 probs_in_mlp: bool = False):
        import torch

        self.moe, self.w, self.dev = moe, w, dev
        self.cfmt = {"bf16": moe.COMBINE_BF16, "mxfp8": moe.COMBINE_MXFP8, "mxfp4": moe.COMBINE_MXFP4}[combine_format]
        if self.cfmt != moe.COMBINE_BF16 and w.dtype != "fp8":
            raise SystemExit("--combine-format mxfp8/mxfp4 is written by the FP8 path's FC2 epilogue only")
        self.combine_format = combine_format
        if probs_in_mlp and w.I == 0:
            raise SystemExit("--probs-in-mlp needs a workload with an expert MLP")
        self.probs_in_mlp = probs_in_mlp
        fmt, rmap, probs = workloads.routing_inputs(w, seed)
        self.fmt = fmt
        self.map_host = torch.from_numpy(np.ascontiguousarray(rmap)).pin_memory()
        self.probs_host = torch.from_numpy(probs).pin_memory()
        self.x_host = workloads.activations(w, seed).pin_memory()
        self.map = self.map_host.to(dev)
        self.probs = self.probs_host.to(dev)
        self.x = self.x_host.to(dev)
        self.identity = w.I == 0
        self.shape = moe.Shape(w.T, w.H, w.E, w.K, w.I)
        self.routing = moe.Routing(fmt, self.map, self.probs)
        # capacity: unbounded, or ceil(rows x factor) 4-aligned from one calibration pass
        cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
        ws = torch.empty(moe.moe_preprocess_workspace_size(self.shape), dtype=torch.uint8, device=dev)
        if w.cap_factor:
            cal_layout = moe.Layout(w.m, cap)
            h = moe.Handle.empty(self.shape, cal_layout, dev)
            moe.moe_preprocess(self.routing, self.shape, cal_layout, h, ws)
            torch.cuda.synchronize()
            cap = moe.moe_capacity(int(h.total_rows.item()), w.cap_factor, 4)
        self.cap = cap
        self.layout = moe.Layout(w.m, cap)
        self.ws = ws
        self.handle = moe.Handle.empty(self.shape, self.layout, dev)
        self.in_dtype = {"bf16": moe.DTYPE_BF16, "fp8": moe.DTYPE_BF16_TO_FP8, "nvfp4": moe.DTYPE_BF16_TO_NVFP4}[w.dtype]
        self.w_dtype = {"bf16": moe.DTYPE_BF16, "fp8": moe.DTYPE_FP8_E4M3_B128, "nvfp4": moe.DTYPE_NVFP4}[w.dtype]
        if w.dtype == "bf16":
            self.y = torch.empty(cap, w.H, dtype=torch.bfloat16, device=dev)
            self.y_scales = None
        elif w.dtype == "fp8":
            self.y = torch.empty(cap, w.H, dtype=torch.uint8, device=dev)
            self.y_scales = torch.empty(cap, w.H // 128, dtype=torch.float32, device=dev)
        else:
            self.y = torch.empty(cap, w.H // 2, dtype=torch.uint8, device=dev)
            self.y_scales = torch.empty(cap, w.H // 16, dtype=torch.uint8, device=dev)
        self.yp = torch.empty(cap, dtype=torch.float32, device=dev)
        self.out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev)
        self.out_host = torch.empty(w.T, w.H, dtype=torch.bfloat16).pin_memory()
        # slot 1 of the double-buffered end-to-end pipeline: its own inputs and output
        map1, probs1 = torch.empty_like(self.map), torch.empty_like(self.probs)
        self.slots = [
            dict(x=self.x, map=self.map, probs=self.probs, routing=self.routing, out=self.out,
                 out_host=self.out_host),
            dict(x=torch.empty_like(self.x), map=map1, probs=probs1, routing=moe.Routing(fmt, map1, probs1),
                 out=torch.empty_like(self.out), out_host=torch.empty_like(self.out_host).pin_memory()),
        ]
        self.globals = None
        self.x_scales = None
        if not self.identity:
            w13, w2 = workloads.expert_weights(w, seed, device=dev)
            if w.dtype == "bf16":
                self.w13, self.w2, self.w13_s, self.w2_s = w13, w2, None, None
            elif w.dtype == "fp8":
                self.w13 = torch.empty(w13.shape, dtype=torch.uint8, device=dev)
                self.w13_s = torch.empty(w.E, 2 * w.I // 128, w.H // 128, dtype=torch.float32, device=dev)
                self.w2 = torch.empty(w2.shape, dtype=torch.uint8, device=dev)
                self.w2_s = torch.empty(w.E, w.H // 128, w.I // 128, dtype=torch.float32, device=dev)
                moe.moe_quantize_fp8_blocks(w13, self.w13, self.w13_s)
                moe.moe_quantize_fp8_blocks(w2, self.w2, self.w2_s)
            else:
                g13 = (w13.float().abs().amax(dim=(1, 2)) / (6 * 448)).contiguous()
                g2 = (w2.float().abs().amax(dim=(1, 2)) / (6 * 448)).contiguous()
                self.w13 = torch.empty(w.E, 2 * w.I, w.H // 2, dtype=torch.uint8, device=dev)
                self.w13_s = torch.empty(w.E, 2 * w.I, w.H // 16, dtype=torch.uint8, device=dev)
                self.w2 = torch.empty(w.E, w.H, w.I // 2, dtype=torch.uint8, device=dev)
                self.w2_s = torch.empty(w.E, w.H, w.I // 16, dtype=torch.uint8, device=dev)
                for e in range(w.E):
                    moe.moe_quantize_nvfp4_rows(w13[e], g13[e:e + 1], self.w13[e], self.w13_s[e])
                    moe.moe_quantize_nvfp4_rows(w2[e], g2[e:e + 1], self.w2[e], self.w2_s[e])
                g1 = (self.x.float().abs().amax() / (6 * 448)).reshape(1)
                self.x_scales = g1
                self.globals = moe.Nvfp4Globals(g1, torch.tensor([0.01], device=dev), g13, g2)
            del w13, w2
            torch.cuda.empty_cache()  # release the bf16 weight temporaries
            self.act_ws = torch.empty(moe.moe_grouped_mlp_workspace_size(self.shape, self.layout, self.w_dtype),
                                      dtype=torch.uint8, device=dev)
            if self.cfmt == moe.COMBINE_BF16:
                self.o = torch.empty(cap, w.H, dtype=torch.bfloat16, device=dev)
                self.o_scales = None
            else:
                self.o = torch.empty(cap, w.H if self.cfmt == moe.COMBINE_MXFP8 else w.H // 2, dtype=torch.uint8,
                                     device=dev)
                self.o_scales = torch.empty(cap, w.H // 32, dtype=torch.uint8, device=dev)
            self.mlp_kernels = moe.moe_grouped_mlp_kernel_count(self.shape, self.layout, self.w_dtype)
        torch.cuda.synchronize()

    def step(self, stream, ev=None, prof=None, slot=0):
        """The four library calls.  ev: events recorded at the call boundaries --
        a list of 5 (before and after every call), or a dict {index: event} for
        a subset of the boundaries 0..4; prof: the grouped-MLP profiling hook's
        three events; slot: which input/output buffer set to use."""
        moe = self.moe
        io = self.slots[slot]
        if isinstance(ev, dict):
            rec = lambda i: ev[i].record(stream) if i in ev else None
        else:
            rec = (lambda i: ev[i].record(stream)) if ev else (lambda i: None)
        rec(0)
        self.call_preprocess(stream, slot)
        rec(1)
        self.call_dispatch(stream, slot)
        rec(2)
        if not self.identity:
            if prof:
                moe.moe_profile_next_grouped_mlp(*prof)
            moe.moe_grouped_mlp_ex(self.handle, self.shape, self.layout, self.w_dtype, self.y, self.y_scales,
                                   self.w13, self.w13_s, self.w2, self.w2_s, self.globals, self.act_ws, self.cfmt,
                                   self.o, self.o_scales, self.yp if self.probs_in_mlp else None, stream=stream)
        rec(3)
        self.call_combine(stream, slot)
        rec(4)

    def call_preprocess(self, stream, slot=0):
        io = self.slots[slot]
        self.moe.moe_preprocess(io["routing"], self.shape, self.layout, self.handle, self.ws, stream=stream)

    def call_dispatch(self, stream, slot=0):
        io = self.slots[slot]
        self.moe.moe_dispatch_permute(self.handle, self.shape, self.layout, self.in_dtype, io["x"], self.x_scales,
                                      io["routing"], self.y, self.yp, self.y_scales, stream=stream)

    def call_combine(self, stream, slot=0):
        io = self.slots[slot]
        if self.identity:
            self.moe.moe_combine_unpermute(self.handle, self.shape, self.layout, self.y, self.yp, io["out"],
                                           stream=stream)
        else:
            # probabilities applied inside the MLP: the combine sums the rows unweighted
            self.moe.moe_combine_unpermute_fmt(self.handle, self.shape, self.layout, self.cfmt, self.o,
                                               self.o_scales, None if self.probs_in_mlp else self.yp, io["out"],
                                               stream=stream)

    def kernels_per_step(self) -> int:
        return 2 + 1 + (0 if self.identity else self.mlp_kernels) + 1

    def routed_rows(self) -> int:
        import torch
        torch.cuda.synchronize()
        return int(self.handle.row_of[: self.w.T * self.w.K].ge(0).sum().item())

    # algorithmic work per launch
    def fc1_flops(self, R):
        return 2.0 * R * self.w.H * 2 * self.w.I

    def fc2_flops(self, R):
        return 2.0 * R * self.w.I * self.w.H

    def active_experts(self) -> int:
        import torch
        torch.cuda.synchronize()
        return int(self.handle.tokens_per_expert.gt(0).sum().item())

    def _elem_bytes(self, n):
        """Bytes of n values stored as bf16, or as NVFP4 (packed E2M1 + one E4M3 scale per 16)."""
        return n / 2 + n / 16 if self.w.dtype == "nvfp4" else 2.0 * n

    def fc1_bytes(self, R, active):
        """FC1 algorithmic bytes: the active experts' w3_w1, the dispatched rows, the intermediate written."""
        w = self.w
        if w.dtype == "fp8":
            wb = 2 * w.I * w.H + 4 * (2 * w.I // 128) * (w.H // 128)
            return active * wb + R * (w.H + 4 * w.H // 128) + R * (w.I + 4 * w.I // 128)
        wb = self._elem_bytes(2 * w.I * w.H)
        return active * wb + R * self._elem_bytes(w.H) + R * self._elem_bytes(w.I)

    def out_row_bytes(self):
        """Bytes of one expert-output row in the combine format."""
        w = self.w
        if getattr(self, "combine_format", "bf16") == "mxfp8":
            return w.H + w.H // 32
        if getattr(self, "combine_format", "bf16") == "mxfp4":
            return w.H // 2 + w.H // 32
        return 2 * w.H

    def fc2_bytes(self, R, active):
        """FC2 algorithmic bytes: the active experts' w2, the intermediate read, the output rows written."""
        w = self.w
        if w.dtype == "fp8":
            wb = w.H * w.I + 4 * (w.H // 128) * (w.I // 128)
            return active * wb + R * (w.I + 4 * w.I // 128) + R * self.out_row_bytes()
        return active * self._elem_bytes(w.H * w.I) + R * self._elem_bytes(w.I) + R * 2 * w.H

    def dispatch_bytes(self, R):
        w = self.w
        row_in = {"bf16": 2 * w.H, "fp8": 2 * w.H, "nvfp4": 2 * w.H}[w.dtype]
        row_out = {"bf16": 2 * w.H, "fp8": w.H + 4 * (w.H // 128), "nvfp4": w.H // 2 + w.H // 16}[w.dtype]
        return w.T * row_in + R * row_out + R * 4 + w.T * w.K * 4 * 2

    def combine_bytes(self, R):
        w = self.w
        return R * self.out_row_bytes() + R * 4 + w.T * w.K * 4 + w.T * 2 * w.H


def make_prof_events(n, stream):
    """n triples of timing events for the grouped-MLP profiling hook, created
    (recorded once) before the library records them."""
    import torch

    trios = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for trio in trios:
        for e in trio:
            e.record(stream)
    return trios


def capture_step_graphs(prob, stream, n):
    """CUDA graphs of one step.  MLP workloads: n captures of the four calls,
    capture i with the profiling hook's event triple i inside (event-record
    nodes), returned as (graphs, triples, None).  Identity experts: one graph
    each of preprocess, dispatch and combine, replayed with n pairs of events
    around the dispatch graph, returned as (graphs, None, pairs)."""
    import torch

    torch.cuda.synchronize()
    if prob.identity:
        parts = []
        for fn in (prob.call_preprocess, prob.call_dispatch, prob.call_combine):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn(stream)
            parts.append(g)
        pairs = [{1: torch.cuda.Event(enable_timing=True), 2: torch.cuda.Event(enable_timing=True)}
                 for _ in range(n)]
        return ("split", parts), None, pairs
    trios = make_prof_events(n, stream)
    torch.cuda.synchronize()
    graphs = []
    for i in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            prob.step(stream, prof=trios[i])
        graphs.append(g)
    torch.cuda.synchronize()
    return ("whole", graphs), trios, None


def replay_step(graphs, i, stream, dev_pair):
    kind, gs = graphs
    if kind == "whole":
        gs[i % len(gs)].replay()
        return
    gs[0].replay()
    if dev_pair:
        dev_pair[1].record(stream)
    gs[1].replay()
    if dev_pair:
        dev_pair[2].record(stream)
    gs[2].replay()


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import __graft_entry__

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # the device first, so that NCCL's communicator and every barrier use this rank's GPU
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    if rank == 0 or world == 1:
        __graft_entry__.build_library()
    if world > 1:
        dist.barrier()
    import permute_grouped_expert_gb300 as moe

    prob = Problem(moe, w, args.seed + rank, dev, args.combine_format, args.probs_in_mlp)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for _ in range(W):
            prob.step(stream)
    torch.cuda.synchronize()

    # ---- device-timed region: inputs resident in HBM; every step is the replay
    # of a CUDA graph of the four library calls.  Events between the replays give
    # each step's time.  The dominant kernel is timed inside the same replays:
    # for MLP workloads the grouped-MLP profiling hook records its events as
    # event-record nodes of the graph, so step i's graph (one capture per step,
    # each with its own events) carries step i's events; for identity experts the
    # step is three graphs (preprocess, dispatch, combine) with events between.
    graphs, pevs, devs = capture_step_graphs(prob, stream, K)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    step_evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    est = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    with torch.cuda.stream(stream):
        est[0].record(stream)
        replay_step(graphs, 0, stream, None)
        est[1].record(stream)
    torch.cuda.synchronize()
    n_pre = pre_roll_count(est[0].elapsed_time(est[1]), W)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(n_pre):  # warm replays of the captured graphs, under the clock sampler
            replay_step(graphs, 0, stream, None)
        for i in range(K):
            step_evs[i].record(stream)
            replay_step(graphs, i, stream, devs[i] if devs else None)
        step_evs[K].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    per_step = [step_evs[i].elapsed_time(step_evs[i + 1]) for i in range(K)]
    total_ms = max_over_ranks(step_evs[0].elapsed_time(step_evs[K]), dev)
    ms_step = total_ms / K

    def stats(xs):
        return {"mean": round(statistics.mean(xs), 5), "min": round(min(xs), 5),
                "median": round(statistics.median(xs), 5)}

    def durations(a, b, table, n):
        return [table[i][a].elapsed_time(table[i][b]) for i in range(n)]

    kernel_timing = "events inside the timed graph replays"
    try:
        fc1_ts = durations(0, 1, pevs, K) if pevs else None
        fc2_ts = durations(1, 2, pevs, K) if pevs else None
    except RuntimeError:
        # the events recorded by graph nodes could not be read: time the grouped
        # MLP's kernels in an eager pass instead (said so in the line)
        kernel_timing = "events around the kernels in an eager pass after the timed region"
        pevs = make_prof_events(K, stream)
        with torch.cuda.stream(stream):
            for i in range(K):
                prob.step(stream, prof=pevs[i])
        torch.cuda.synchronize()
        fc1_ts, fc2_ts = durations(0, 1, pevs, K), durations(1, 2, pevs, K)
    dis_ts = durations(1, 2, devs, K) if devs else None
    t_fc1 = statistics.mean(fc1_ts) if fc1_ts else None
    t_fc2 = statistics.mean(fc2_ts) if fc2_ts else None
    t_dis_timed = statistics.mean(dis_ts) if dis_ts else None

    # ---- per-call breakdown: a separate eager pass with events at every call boundary
    KB = min(K, 50)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(KB)]
    with torch.cuda.stream(stream):
        for i in range(KB):
            prob.step(stream, evs[i])
    torch.cuda.synchronize()
    call_ts = {name: durations(a, a + 1, evs, KB) for a, name in
               enumerate(("preprocess", "dispatch", "grouped_mlp", "combine"))}
    t_pre = statistics.mean(call_ts["preprocess"])
    t_dis = t_dis_timed if devs else statistics.mean(call_ts["dispatch"])
    t_mlp = statistics.mean(call_ts["grouped_mlp"])
    t_com = statistics.mean(call_ts["combine"])

    # ---- end to end: every step copies its inputs in from pinned host memory
    # and its layer output back out.  Two buffer slots and two copy streams let
    # step i+1's inputs and step i-1's output move while step i computes, as a
    # serving loop would run it.
    e2e_evs = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    h2d = prob.x_host.numel() * 2 + prob.map_host.numel() * prob.map_host.element_size() + prob.probs_host.numel() * 4
    d2h = prob.out_host.numel() * 2
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    compute_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    last_out = torch.cuda.Event()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e2e_clocks = ClockSampler(clocks.gpu)
    e2e_clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(n_pre):  # load under the sampler's first samples
            replay_step(graphs, 0, stream, None)
    e2e_evs[0].record(stream)
    cin.wait_event(e2e_evs[0])
    for i in range(K):
        sl = i % 2
        io = prob.slots[sl]
        if i >= 2:
            cin.wait_event(compute_done[sl])  # step i-2 no longer reads this slot's inputs
        with torch.cuda.stream(cin):
            io["x"].copy_(prob.x_host, non_blocking=True)
            io["map"].copy_(prob.map_host, non_blocking=True)
            io["probs"].copy_(prob.probs_host, non_blocking=True)
            in_done[sl].record(cin)
        stream.wait_event(in_done[sl])
        if i >= 2:
            stream.wait_event(out_done[sl])  # step i-2's output has left this slot
        with torch.cuda.stream(stream):
            prob.step(stream, slot=sl)
            compute_done[sl].record(stream)
        cout.wait_event(compute_done[sl])
        with torch.cuda.stream(cout):
            io["out_host"].copy_(io["out"], non_blocking=True)
            out_done[sl].record(cout)
    last_out.record(cout)
    stream.wait_event(last_out)
    e2e_evs[1].record(stream)
    torch.cuda.synchronize()
    e2e_clk = e2e_clocks.stop()
    e2e_ms = max_over_ranks(e2e_evs[0].elapsed_time(e2e_evs[1]), dev)

    R = prob.routed_rows()
    overflow = int(prob.handle.overflow.item())
    status = int(prob.handle.status.item())
    tokens = w.T * world
    value = job_throughput(w.T, world, K, total_ms)
    peaks, peak_src = load_peaks()

    breakdown = {
        "step_ms": stats(per_step), "timing": "each step one CUDA graph replay of the four calls; "
        + ("dispatch timed by events between the preprocess, dispatch and combine graphs" if prob.identity
           else "grouped-MLP kernels timed by " + kernel_timing),
        "calls_ms": {k: stats(v) for k, v in call_ts.items() if not (prob.identity and k == "grouped_mlp")},
        "preprocess_ms": round(t_pre, 5), "dispatch_ms": round(t_dis, 5), "combine_ms": round(t_com, 5),
        "dispatch_gbs": round(prob.dispatch_bytes(R) / (t_dis * 1e-3) / 1e9, 1),
        "combine_gbs": round(prob.combine_bytes(R) / (t_com * 1e-3) / 1e9, 1),
        "routed_rows": R, "capacity": prob.cap, "overflow": overflow, "device_status": status,
    }
    if prob.identity:
        dom = "dispatch_permute"
        achieved = prob.dispatch_bytes(R) / (t_dis * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": profiled_traffic(w.name, "permute_grouped_expert_gb300/csrc/permute.cu"),
                "peak_source": f"{peak_src} hbm_gbs"}
    else:
        peak = peaks["bf16_tflops"] * (2.0 if w.dtype == "fp8" else 4.0 if w.dtype == "nvfp4" else 1.0)
        peak_source = f"{peak_src} bf16_tflops (burst)" + (" x nominal dtype ratio" if w.dtype != "bf16" else "")
        breakdown["grouped_mlp_ms"] = round(t_mlp, 5)
        if prob.mlp_kernels == 1:
            # FC1, SwiGLU and FC2 in one persistent kernel: its roofline counts both GEMMs
            flops = prob.fc1_flops(R) + prob.fc2_flops(R)
            achieved = flops / (t_fc1 * 1e-3) / 1e12
            breakdown.update({"fused_mlp_kernel_ms": stats(fc1_ts), "fused_mlp_tflops": round(achieved, 1)})
            kernel = "grouped_mlp_bf16 (FC1 + SwiGLU + FC2, one kernel)"
            traffic = profiled_traffic(w.name, "permute_grouped_expert_gb300/csrc/gemm_bf16.cu")
        elif w.dtype == "nvfp4":
            # decode: a few rows per expert, so FC1 streams the active experts' weights (HBM-bound)
            active = prob.active_experts()
            fc1_bytes = prob.fc1_bytes(R, active)
            achieved_gbs = fc1_bytes / (t_fc1 * 1e-3) / 1e9
            breakdown.update({"fc1_ms": stats(fc1_ts), "fc2_ms": stats(fc2_ts), "active_experts": active,
                              "fc1_tflops": round(prob.fc1_flops(R) / (t_fc1 * 1e-3) / 1e12, 2),
                              "fc1_weight_gbs": round(achieved_gbs, 1),
                              "fc2_weight_gbs": round(prob.fc2_bytes(R, active) / (t_fc2 * 1e-3) / 1e9, 1)})
            roof = {"kernel": "grouped_fc1_swiglu (NVFP4)", "bound": "hbm", "achieved": round(achieved_gbs, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
                    "traffic": profiled_traffic(w.name, "permute_grouped_expert_gb300/csrc/gemm_nvfp4.cu"),
                    "peak_source": f"{peak_src} hbm_gbs"}
            kernel = None
        else:
            achieved = prob.fc1_flops(R) / (t_fc1 * 1e-3) / 1e12
            breakdown.update({"fc1_ms": stats(fc1_ts), "fc2_ms": stats(fc2_ts),
                              "fc1_tflops": round(achieved, 1),
                              "fc2_tflops": round(prob.fc2_flops(R) / (t_fc2 * 1e-3) / 1e12, 1),
                              "fc2_frac_of_peak": round(prob.fc2_flops(R) / (t_fc2 * 1e-3) / 1e12 / peak, 4)})
            kernel = "grouped_fc1_swiglu"
            traffic = None
            if w.dtype == "fp8":
                # FC1 is bounded by max(FLOPs / FP8 peak, its bytes / HBM): report the
                # fraction against whichever bound is larger, with both fractions beside it
                active = prob.active_experts()
                fc1_b, fc2_b = prob.fc1_bytes(R, active), prob.fc2_bytes(R, active)
                t_flop = prob.fc1_flops(R) / (peak * 1e12)
                t_byte = fc1_b / (peaks["hbm_gbs"] * 1e9)
                gbs = fc1_b / (t_fc1 * 1e-3) / 1e9
                breakdown.update({
                    "active_experts": active,
                    "fc1_weight_hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                    "fc2_weight_hbm_frac": round(fc2_b / (t_fc2 * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                    "fc2_frac_of_max_bound": round(max(prob.fc2_flops(R) / (peak * 1e12),
                                                       fc2_b / (peaks["hbm_gbs"] * 1e9)) / (t_fc2 * 1e-3), 4)})
                traffic = profiled_traffic(w.name, "permute_grouped_expert_gb300/csrc/gemm_fp8.cu")
                if t_byte >= t_flop:
                    roof = {"kernel": "grouped_fc1_swiglu (FP8)", "bound": "hbm", "achieved": round(gbs, 1),
                            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                            "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs",
                            "tensor_frac": round(achieved / peak, 4),
                            "note": "max(FLOPs / FP8 peak, bytes / HBM) binds on bytes: "
                                    f"{t_byte * 1e3:.3f} ms vs {t_flop * 1e3:.3f} ms"}
                    kernel = None
        if kernel is not None:
            roof = {"kernel": kernel, "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                    "peak_source": peak_source}
        roof["launch_ms"] = round(t_fc1, 5)
    if prob.identity:
        roof["launch_ms"] = round(t_dis, 5)
    breakdown["dispatch_frac_of_hbm"] = round(breakdown["dispatch_gbs"] / peaks["hbm_gbs"], 4)
    breakdown["combine_frac_of_hbm"] = round(breakdown["combine_gbs"] / peaks["hbm_gbs"], 4)

    # bytes one step moves through HBM (algorithmic): L2 cannot hold them between steps
    in_bytes = prob.dispatch_bytes(R) + prob.combine_bytes(R) + (0 if prob.identity else sum(
        t.numel() * t.element_size() for t in (prob.w13, prob.w2)))
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded; shapes of the pages' workloads)",
        "config": {"workload": w.name, "tokens": w.T, "hidden": w.H, "experts": w.E, "topk": w.K,
                   "intermediate": w.I, "pad_multiple": w.m, "routing": w.routing,
                   "combine_format": args.combine_format,
                   "probs_applied": "in the MLP (FC2 epilogue)" if args.probs_in_mlp else "in the combine",
                   "capacity_factor": w.cap_factor or None, "capacity": prob.cap,
                   "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB moved per step vs {L2_BYTES / 1e6:.0f} MB L2)"
                   if in_bytes > L2_BYTES else "inputs smaller than L2 (no flush)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "breakdown": breakdown,
        "e2e": {"value": round(job_throughput(w.T, world, K, e2e_ms), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / K, 5), "clocks": e2e_clk},
        "gpu_launches": prob.kernels_per_step() * K,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.seed, sample_tokens=args.cpu_sample_tokens,
                                            target_s=args.cpu_seconds, probs_in_mlp=args.probs_in_mlp)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------- backward

class BackwardProblem:
    """Buffers of the layer's backward through combine and dispatch: the combine
    backward (gradient row per route, probability gradient per row) then the
    dispatch backward (token gradients, probability gradients in the routing
    layout).  The expert MLP's own backward is not part of this path, so the
    dispatch backward takes the combine backward's row gradients as the
    gradients of the dispatched rows (the whole layer's backward for identity
    experts).  The forward state it needs -- the handle, the dispatched
    probabilities and the expert rows -- comes from one forward step of `prob`."""

    def __init__(self, prob, seed):
        import torch

        moe, w, dev = prob.moe, prob.w, prob.dev
        if not prob.identity and prob.cfmt != moe.COMBINE_BF16:
            raise SystemExit("--direction backward reads bf16 expert rows (--combine-format bf16)")
        if prob.identity and w.dtype != "bf16":
            raise SystemExit("--direction backward with identity experts needs bf16 rows")
        self.prob, self.moe, self.w = prob, moe, w
        self.o = prob.y if prob.identity else prob.o
        self.gy_host = workloads.grad_outputs(w, seed).pin_memory()
        self.gy = self.gy_host.to(dev)
        cap = prob.cap
        self.g_o = torch.empty(cap, w.H, dtype=torch.bfloat16, device=dev)
        self.g_w = torch.empty(cap, dtype=torch.float32, device=dev)
        self.g_x = torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev)
        gp_shape = (w.T, w.K) if prob.fmt == moe.ROUTING_DENSE_I16 else (w.T, w.E)
        self.g_p = torch.empty(gp_shape, dtype=torch.float32, device=dev)
        self.slots = [dict(gy=self.gy, g_x=self.g_x, g_p=self.g_p,
                           g_x_host=torch.empty(self.g_x.shape, dtype=torch.bfloat16).pin_memory(),
                           g_p_host=torch.empty(gp_shape, dtype=torch.float32).pin_memory()),
                      dict(gy=torch.empty_like(self.gy), g_x=torch.empty_like(self.g_x), g_p=torch.empty_like(self.g_p),
                           g_x_host=torch.empty(self.g_x.shape, dtype=torch.bfloat16).pin_memory(),
                           g_p_host=torch.empty(gp_shape, dtype=torch.float32).pin_memory())]

    def call_combine_backward(self, stream, slot=0):
        p = self.prob
        self.moe.moe_combine_backward(p.handle, p.shape, p.layout, self.slots[slot]["gy"], self.o, p.yp, self.g_o,
                                      self.g_w, stream=stream)

    def call_dispatch_backward(self, stream, slot=0):
        p, io = self.prob, self.slots[slot]
        self.moe.moe_dispatch_backward(p.handle, p.shape, p.layout, p.fmt, self.g_o, self.g_w, io["g_x"],
                                       io["g_p"], stream=stream)

    def step(self, stream, ev=None, slot=0):
        if ev:
            ev[0].record(stream)
        self.call_combine_backward(stream, slot)
        if ev:
            ev[1].record(stream)
        self.call_dispatch_backward(stream, slot)
        if ev:
            ev[2].record(stream)

    kernels_per_step = 3  # combine backward; dispatch backward = weight-1 combine + probability-gradient gather

    def valid_rows(self):
        import torch
        torch.cuda.synchronize()
        return min(int(self.prob.handle.total_rows.item()), self.prob.cap)

    def combine_backward_bytes(self, R, V):
        """gy read once, the routed expert rows read, gradient rows written for
        routed and pad rows, one probability gradient per row, the row map and
        the dispatched probabilities read."""
        w = self.w
        return w.T * w.H * 2 + R * w.H * 2 + V * w.H * 2 + V * 4 + R * 4 + w.T * w.K * 4

    def dispatch_backward_bytes(self, R):
        """Gradient rows read, token gradients written, the row map read twice,
        row probability gradients read and written into the routing layout."""
        w = self.w
        return R * w.H * 2 + w.T * w.H * 2 + 2 * w.T * w.K * 4 + R * 4 + self.g_p.numel() * 4


def run_backward(args, w):
    import torch

    import __graft_entry__

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    if rank == 0 or world == 1:
        __graft_entry__.build_library()
    if world > 1:
        dist.barrier()
    import permute_grouped_expert_gb300 as moe

    prob = Problem(moe, w, args.seed + rank, dev, args.combine_format, args.probs_in_mlp)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        prob.step(stream)  # the forward state the backward reads
    torch.cuda.synchronize()
    bp = BackwardProblem(prob, args.seed + rank)
    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for _ in range(W):
            bp.step(stream)
    torch.cuda.synchronize()

    # ---- device-timed region: two graphs per step (combine backward, dispatch
    # backward) with events between them, inputs resident in HBM
    graphs = []
    for fn in (bp.call_combine_backward, bp.call_dispatch_backward):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn(stream)
        graphs.append(g)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    est = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    with torch.cuda.stream(stream):
        est[0].record(stream)
        graphs[0].replay()
        graphs[1].replay()
        est[1].record(stream)
    torch.cuda.synchronize()
    n_pre = pre_roll_count(est[0].elapsed_time(est[1]), W)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(n_pre):  # warm replays under the clock sampler
            graphs[0].replay()
            graphs[1].replay()
        for i in range(K):
            evs[i][0].record(stream)
            graphs[0].replay()
            evs[i][1].record(stream)
            graphs[1].replay()
            evs[i][2].record(stream)
        end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = max_over_ranks(evs[0][0].elapsed_time(end), dev)
    ms_step = total_ms / K
    t_cb = [evs[i][0].elapsed_time(evs[i][1]) for i in range(K)]
    t_db = [evs[i][1].elapsed_time(evs[i][2]) for i in range(K)]

    # ---- end to end: each step copies dL/dy in from pinned host memory and the
    # token and probability gradients back out (two slots, two copy streams)
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    compute_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    e0, e1, last_out = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                        torch.cuda.Event())
    h2d = bp.gy_host.numel() * 2
    d2h = bp.g_x.numel() * 2 + bp.g_p.numel() * 4
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e2e_clocks = ClockSampler(clocks.gpu)
    e2e_clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(n_pre):  # load under the sampler's first samples
            graphs[0].replay()
            graphs[1].replay()
    e0.record(stream)
    cin.wait_event(e0)
    for i in range(K):
        sl = i % 2
        io = bp.slots[sl]
        if i >= 2:
            cin.wait_event(compute_done[sl])
        with torch.cuda.stream(cin):
            io["gy"].copy_(bp.gy_host, non_blocking=True)
            in_done[sl].record(cin)
        stream.wait_event(in_done[sl])
        if i >= 2:
            stream.wait_event(out_done[sl])
        with torch.cuda.stream(stream):
            bp.step(stream, slot=sl)
            compute_done[sl].record(stream)
        cout.wait_event(compute_done[sl])
        with torch.cuda.stream(cout):
            io["g_x_host"].copy_(io["g_x"], non_blocking=True)
            io["g_p_host"].copy_(io["g_p"], non_blocking=True)
            out_done[sl].record(cout)
    last_out.record(cout)
    stream.wait_event(last_out)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_clk = e2e_clocks.stop()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)

    R = prob.routed_rows()
    V = bp.valid_rows()
    peaks, peak_src = load_peaks()
    cb_gbs = bp.combine_backward_bytes(R, V) / (statistics.mean(t_cb) * 1e-3) / 1e9
    db_gbs = bp.dispatch_backward_bytes(R) / (statistics.mean(t_db) * 1e-3) / 1e9

    def stats(xs):
        return {"mean": round(statistics.mean(xs), 5), "min": round(min(xs), 5),
                "median": round(statistics.median(xs), 5)}

    cb_dominant = statistics.mean(t_cb) >= statistics.mean(t_db)
    achieved = cb_gbs if cb_dominant else db_gbs
    roof = {"kernel": "combine_backward" if cb_dominant else "dispatch_backward (weight-1 combine + gather)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": profiled_traffic(w.name + ":backward", "permute_grouped_expert_gb300/csrc/backward.cu"),
            "peak_source": f"{peak_src} hbm_gbs",
            "launch_ms": round(statistics.mean(t_cb if cb_dominant else t_db), 5)}
    in_bytes = bp.combine_backward_bytes(R, V) + bp.dispatch_backward_bytes(R)
    line = {
        "metric": METRIC, "value": round(job_throughput(w.T, world, K, total_ms), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the pages' workloads)",
        "config": {"workload": w.name, "direction": "backward (combine backward + dispatch backward)",
                   "tokens": w.T, "hidden": w.H, "experts": w.E, "topk": w.K, "intermediate": w.I,
                   "pad_multiple": w.m, "routing": w.routing, "capacity": prob.cap,
                   "expert_backward": "not part of the path: the dispatch backward takes the combine backward's "
                                      "row gradients" if not prob.identity else "identity experts",
                   "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB moved per step vs {L2_BYTES / 1e6:.0f} MB L2)"
                   if in_bytes > L2_BYTES else "inputs smaller than L2 (no flush)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "breakdown": {"combine_backward_ms": stats(t_cb), "dispatch_backward_ms": stats(t_db),
                      "combine_backward_gbs": round(cb_gbs, 1), "dispatch_backward_gbs": round(db_gbs, 1),
                      "combine_backward_frac_of_hbm": round(cb_gbs / peaks["hbm_gbs"], 4),
                      "dispatch_backward_frac_of_hbm": round(db_gbs / peaks["hbm_gbs"], 4),
                      "routed_rows": R, "valid_rows": V,
                      "timing": "each step two CUDA graph replays (combine backward, dispatch backward) with "
                                "events between them"},
        "e2e": {"value": round(job_throughput(w.T, world, K, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / K, 5),
                "clocks": e2e_clk},
        "gpu_launches": bp.kernels_per_step * K,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_backward(BackwardOracleInputs(w, args.seed), target_s=args.cpu_seconds)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


class BackwardOracleInputs:
    """The oracle-side inputs of the backward, prepared once (not timed): the
    routing, its preprocess, the expert rows (the oracle's dispatch of the
    activations, standing in for the expert outputs: the cost does not depend
    on the values) and dL/dy."""

    def __init__(self, w, seed):
        import oracle

        oracle.build()
        self.w = w
        self.fmt, self.rmap, probs = workloads.routing_inputs(w, seed)
        cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
        if w.cap_factor:
            cap = oracle.capacity(oracle.preprocess(self.fmt, self.rmap, w.T, w.E, w.K, w.m, cap)["total_rows"],
                                  w.cap_factor)
        self.pre = oracle.preprocess(self.fmt, self.rmap, w.T, w.E, w.K, w.m, cap)
        self.o, self.po = oracle.dispatch(self.fmt, self.rmap, probs, self.pre,
                                          workloads.bf16_bits(workloads.activations(w, seed)), cap, w.E, w.K)
        self.gy = workloads.bf16_bits(workloads.grad_outputs(w, seed))


def cpu_baseline_backward(inp, target_s=None, sample_tokens=64):
    """The oracle's combine and dispatch backward as they stand, on a bounded
    sample: batches of tokens (all their routes) until target_s seconds (or
    sample_tokens tokens without a target), extrapolated to the batch.  Each
    batch's rows are renumbered onto a compact list (the oracle's outputs are
    sized by the rows it is given)."""
    import oracle

    w = inp.w
    order = np.random.default_rng(0).permutation(w.T)
    done, t = 0, 0.0
    n = 1 if target_s is not None else sample_tokens
    while done < w.T:
        n = min(n, w.T - done)
        toks = np.sort(order[done:done + n])
        row_of = inp.pre["row_of"][toks]
        sel = np.unique(row_of[row_of >= 0])
        local = np.where(row_of >= 0, np.searchsorted(sel, np.where(row_of >= 0, row_of, 0)), -1).astype(np.int32)
        sub = {"row_of": local, "counts": np.array([len(sel)], np.int32),
               "offsets": np.array([0, len(sel)], np.int32)}
        o_sel, po_sel, gy_sel, map_sel = inp.o[sel], inp.po[sel], inp.gy[toks], np.ascontiguousarray(inp.rmap[toks])
        t0 = time.perf_counter()
        g_o, g_w = oracle.combine_backward(gy_sel, sub, len(sel), o_sel, po_sel)
        oracle.dispatch_backward(inp.fmt, map_sel, local, w.E, g_o, g_w)
        t += time.perf_counter() - t0
        done += n
        if target_s is None or t >= target_s:
            break
        per_token = t / done
        n = max(1, min(2 * done, int((target_s - t) / max(per_token, 1e-9)) + 1))
    return {"value": round(done / t, 2), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"combine backward + dispatch backward of {done} sampled tokens ({t:.2f} s) extrapolated "
                      f"x{w.T / done:.1f}; routing preprocess, the row renumbering and input generation not timed"}


# ----------------------------------------------------------- CPU oracle arm

def _nvfp4_global(a) -> float:
    """fp32 global scale amax / (6 * 448) of a tensor (the value the GPU side computes on the host too)."""
    return float(np.float32(float(np.abs(np.asarray(a, np.float32)).max()) / 2688.0))


class OracleWeights:
    """Expert weights in the oracle's format, generated and quantized expert by
    expert on first use and kept: the GPU path prepares its weights once before
    timing, so the oracle's timed sample excludes that preparation too."""

    def __init__(self, w, seed):
        self.w, self.seed, self.cache = w, seed, {}

    def get(self, experts):
        import oracle

        w = self.w
        for e in experts:
            if e in self.cache:
                continue
            w13, w2 = workloads.expert_weights(w, self.seed, experts=[e])
            w13b, w2b = workloads.bf16_bits(w13), workloads.bf16_bits(w2)
            if w.dtype == "fp8":
                self.cache[e] = oracle.quantize_fp8_weight(w13b) + oracle.quantize_fp8_weight(w2b) + (None, None)
            elif w.dtype == "nvfp4":
                g13, g2 = _nvfp4_global(w13.float().numpy()), _nvfp4_global(w2.float().numpy())
                self.cache[e] = (oracle.quantize_nvfp4_rows(w13b, g13) + oracle.quantize_nvfp4_rows(w2b, g2)
                                 + (g13, g2))
            else:
                self.cache[e] = (w13b, None, w2b, None, None, None)
        parts = [self.cache[e] for e in experts]

        def stack(j):
            return None if parts[0][j] is None else np.concatenate([p[j] for p in parts])

        g = None if parts[0][4] is None else (np.array([p[4] for p in parts], np.float32),
                                             np.array([p[5] for p in parts], np.float32))
        return stack(0), stack(1), stack(2), stack(3), g


def cpu_baseline(w, seed, sample_tokens=16, target_s=None, weights=None, probs_in_mlp=False):
    """The oracle as it stands, on a bounded sample: full preprocess and dispatch
    (with the activation quantization of FP8 / NVFP4 workloads; they scale with
    T), then the MLP and combine for sampled tokens (all their routes),
    extrapolated to the whole batch.  Input generation and the expert weights'
    generation and quantization (a one-time preparation on the GPU side too)
    are outside the timed parts.  Without target_s the sample is
    `sample_tokens` tokens; with it, batches of new tokens (starting at one and
    growing with the measured rate) are added until the sampled part has taken
    target_s seconds or every token is in.  probs_in_mlp: the MLP scales its FC2
    rows by the probabilities and the combine sums them unweighted.  Returns the
    cpu_baseline object."""
    import oracle

    oracle.build()
    cores = os.cpu_count()
    weights = weights or OracleWeights(w, seed)
    fmt, rmap, probs = workloads.routing_inputs(w, seed)
    x_t = workloads.activations(w, seed)
    x = workloads.bf16_bits(x_t)
    # FP8 / NVFP4: the activation quantization is per token, so it is sampled
    # with the MLP and combine; the full dispatch copies row buffers of the
    # quantized format (a copy's cost does not depend on the bytes), and each
    # sampled token's quantized row is then placed where that copy put it.
    gx = _nvfp4_global(x_t.float().numpy()) if w.dtype == "nvfp4" else 0.0
    if w.dtype == "fp8":
        xq, xs = np.zeros((w.T, w.H), np.uint8), np.ones((w.T, w.H // 128), np.float32)
    elif w.dtype == "nvfp4":
        xq, xs = np.zeros((w.T, w.H // 2), np.uint8), np.zeros((w.T, w.H // 16), np.uint8)
    else:
        xq, xs = x, None
    t0 = time.perf_counter()
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    if w.cap_factor:
        cap = oracle.capacity(oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)["total_rows"], w.cap_factor)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    yq, yp = oracle.dispatch(fmt, rmap, probs, pre, xq, cap, w.E, w.K)
    ys = oracle.dispatch(fmt, rmap, None, pre, xs, cap, w.E, w.K)[0] if xs is not None else None
    t_full = time.perf_counter() - t0

    order = np.random.default_rng(0).permutation(w.T)
    done, t_sample = 0, 0.0
    n = 1 if target_s is not None else sample_tokens
    fmt_mlp = {"bf16": 0, "fp8": 1, "nvfp4": 2}[w.dtype]
    while done < w.T:
        n = min(n, w.T - done)
        toks = order[done:done + n]
        row_of = pre["row_of"][toks]
        rows = np.unique(row_of[row_of >= 0])
        # untimed bookkeeping: the sampled rows' experts, their weights, and the
        # sampled tokens' row map renumbered onto the compact list of those rows
        experts = sorted({int(np.searchsorted(pre["offsets"], r, side="right") - 1) for r in rows})
        if w.I:
            w13q, s13, w2q, s2, g = weights.get(experts)
            extra = {} if g is None else dict(w13_global=g[0], w2_global=g[1], fc1_in_global=gx,
                                              fc2_in_global=float(np.float32(0.01)))
            sel, off = [], [0]
            for e in experts:
                rr = rows[(rows >= pre["offsets"][e]) & (rows < pre["offsets"][e + 1])]
                sel.append(rr)
                off.append(off[-1] + len(rr))
            sel = np.concatenate(sel)
        else:
            sel = rows
        pos = np.searchsorted(sel, np.where(row_of >= 0, row_of, 0))
        local_row_of = np.where(row_of >= 0, pos, -1).astype(np.int32)
        local_probs = yp[sel]
        t1 = time.perf_counter()
        if w.dtype in ("fp8", "nvfp4"):
            qb, sb = (oracle.quantize_fp8_rows(x[toks]) if w.dtype == "fp8"
                      else oracle.quantize_nvfp4_rows(x[toks], gx))
            t_sample += time.perf_counter() - t1
            for j in range(w.K):  # untimed: the rows the full dispatch already copied
                keep = row_of[:, j] >= 0
                yq[row_of[keep, j]] = qb[keep]
                ys[row_of[keep, j]] = sb[keep]
            t1 = time.perf_counter()
        if w.I:
            ob, _ = oracle.grouped_mlp_rows(fmt_mlp, yq[sel], None if ys is None else ys[sel], w.H, w.I,
                                            len(experts), np.array(off, np.int32), w13q, s13, w2q, s2,
                                            np.arange(len(sel)), row_probs=local_probs if probs_in_mlp else None,
                                            **extra)
        else:
            ob = yq[sel]
        oracle.combine(ob, local_row_of, None if probs_in_mlp else local_probs)
        t_sample += time.perf_counter() - t1
        done += n
        if target_s is None or t_sample >= target_s:
            break
        # next batch: what the rate so far says is left to reach target_s, at most doubling
        per_token = t_sample / done
        n = max(1, min(2 * done, sample_tokens * 64, int((target_s - t_sample) / max(per_token, 1e-9)) + 1))
    est = t_full + t_sample * (w.T / done)
    return {"value": round(w.T / est, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"full preprocess + dispatch of {w.T} tokens ({t_full:.2f} s); "
                      + ("activation quantization, " if w.dtype != "bf16" else "")
                      + f"grouped MLP + combine of {done} sampled tokens ({t_sample:.2f} s) extrapolated "
                      f"x{w.T / done:.1f}; input and expert-weight generation and weight quantization not timed"}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    K, W = args.steps, args.warmup
    if args.direction == "backward":
        run_reference_backward(args, w)
        return
    weights = OracleWeights(w, args.seed)
    for _ in range(W):
        cpu_baseline(w, args.seed, sample_tokens=args.ref_sample_tokens, weights=weights,
                     probs_in_mlp=args.probs_in_mlp)
    vals = []
    t0 = time.perf_counter()
    for _ in range(K):
        vals.append(cpu_baseline(w, args.seed, sample_tokens=args.ref_sample_tokens, weights=weights,
                                 probs_in_mlp=args.probs_in_mlp))
    wall = time.perf_counter() - t0
    v = statistics.mean(x["value"] for x in vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": K, "warmup": W,
            "ms_per_step": round(w.T / v * 1e3, 3),
            "timing": "each step runs the oracle on a bounded sample of the batch (full preprocess and dispatch, "
                      "the MLP and combine of sampled tokens); value and ms_per_step are extrapolated from that "
                      "sample to the whole batch, so ms_per_step x steps exceeds the run's wall time",
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; shapes of the pages' workloads)",
            "config": {"workload": w.name, "tokens": w.T, "hidden": w.H, "experts": w.E, "topk": w.K,
                       "intermediate": w.I,
                       "probs_applied": "in the MLP (FC2 epilogue)" if args.probs_in_mlp else "in the combine"},
            "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s", "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": vals[0]["sample"] + f"; {K} timed samples, {wall:.1f} s wall"},
            "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_backward(args, w):
    """The reference arm of the backward: the oracle's combine and dispatch
    backward, each step a bounded sample of the batch's tokens."""
    K, W = args.steps, args.warmup
    inp = BackwardOracleInputs(w, args.seed)
    for _ in range(W):
        cpu_baseline_backward(inp, sample_tokens=args.ref_sample_tokens)
    t0 = time.perf_counter()
    vals = [cpu_baseline_backward(inp, sample_tokens=args.ref_sample_tokens) for _ in range(K)]
    wall = time.perf_counter() - t0
    v = statistics.mean(x["value"] for x in vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": K, "warmup": W,
            "ms_per_step": round(w.T / v * 1e3, 3),
            "timing": "each step runs the oracle's combine and dispatch backward on a bounded sample of the "
                      "batch's tokens; value and ms_per_step are extrapolated to the whole batch",
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; shapes of the pages' workloads)",
            "config": {"workload": w.name, "direction": "backward (combine backward + dispatch backward)",
                       "tokens": w.T, "hidden": w.H, "experts": w.E, "topk": w.K, "intermediate": w.I},
            "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s", "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": vals[0]["sample"] + f"; {K} timed samples, {wall:.1f} s wall"},
            "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=None, choices=sorted(workloads.WORKLOADS),
                    help="default: dsv3 forward, permute backward")
    ap.add_argument("--direction", default="forward", choices=["forward", "backward"],
                    help="backward: the combine backward and the dispatch backward (the expert MLP's own "
                         "backward is not part of the path)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--combine-format", default="bf16", choices=["bf16", "mxfp8", "mxfp4"],
                    help="format of the expert-output rows the combine reads (MX formats: FP8 path only)")
    ap.add_argument("--probs-in-mlp", action="store_true",
                    help="apply the routing probabilities in the MLP's FC2 epilogue; the combine sums unweighted")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=16, help="batch-size scale of the CPU oracle sample")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="the CPU oracle baseline samples batches until its MLP + combine part took this long")
    ap.add_argument("--ref-sample-tokens", type=int, default=16,
                    help="tokens the reference arm (the CPU oracle) runs through the MLP per timed step")
    ap.add_argument("--set", action="append", default=[], metavar="FIELD=INT",
                    help="shrink the workload for profiling captures, e.g. --set E=32 --set T=1024")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload is None:
        args.workload = "permute" if args.direction == "backward" else "dsv3"
    w = workloads.WORKLOADS[args.workload]
    if args.set:
        changes = {k: int(v) for k, v in (kv.split("=", 1) for kv in args.set)}
        w = workloads.scaled(w, name=w.name + "+" + ",".join(args.set), **changes)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.direction == "backward":
        run_backward(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
