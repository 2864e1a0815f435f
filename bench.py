#!/usr/bin/env python3
"""Benchmark: ms per optimizer update (owner-routed reduce + clip + AdamW).

One step = one whole update over one batch of synthetic gradients: every
microbatch's reduction of all buckets (grs_reduce_all, norm partials fused
on the last microbatch), the global-norm finish (grs_grad_norm_sq) and the
fused clip + AdamW + bf16 cast (grs_clip_adamw_step).  Inputs are resident
in HBM and larger than L2 (each rank's gradient buffer alone exceeds it).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload N]
  python bench.py --impl reference ...   (the CPU oracle, timed on host cores)

Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: the
path has no cross-GPU exchange on one GPU per job.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "ms per optimizer update (reduce+clip+AdamW)"
UNIT = "ms/update"


def mandatory_bytes(buckets, n_micro: int, grad_bytes: int = 2) -> dict:
    """Algorithmic bytes of one update, per kernel, from the bucket geometry
    (one dict per bucket: copies, padded, group_size = R_e, the ranks reduced
    per output element: R for REPLICA_AVG/PARTIAL_SUM, dp for LOCAL_SHARD, 1
    for ALREADY_REDUCED).  Per unique padded element: the reduction reads
    grad_bytes*M*R_e and writes acc 4 (first microbatch) or reads+writes it 8
    (later ones); the update reads acc, master, m, v (16) and writes master,
    m, v (12) and the bf16 parameter (2)."""
    red = upd = last = 0
    for d in buckets:
        elems = int(d["copies"]) * int(d["padded"])
        ge = int(d["group_size"])
        red += elems * (grad_bytes * n_micro * ge + 4 + 8 * (n_micro - 1))
        upd += 30 * elems
        last += elems * (grad_bytes * ge + (4 if n_micro == 1 else 8))
    return {"reduce": red, "update": upd, "total": red + upd, "reduce_last_mb": last}


def variant_bytes(buckets, n_micro: int, grad_bytes: int, n_state_pad: int, n_unique: int,
                  idle=None, idle_rows=None) -> dict:
    """mandatory_bytes for an update where `idle` elements (None: none)
    belong to tensors without a gradient, idle_rows[b] of them in each state
    row of bucket b.  Those need no reduction and no update.  The norm, plain
    or masked, is fused into the last reduction (0 bytes); a separate masked
    norm pass would read acc once (4 bytes per element of a tensor with a
    gradient, `norm_pass`)."""
    mb = mandatory_bytes(buckets, n_micro, grad_bytes)
    mb["norm"] = 0
    if idle is not None:
        if idle_rows is not None:
            live_b = [dict(d, padded=int(d["padded"]) - int(r)) for d, r in zip(buckets, idle_rows)]
            mb["reduce"] = mandatory_bytes(live_b, n_micro, grad_bytes)["reduce"]
        live = n_state_pad - idle          # elements the update writes (padding included)
        mb["norm_pass"] = 4 * (n_unique - idle)  # elements a separate norm pass reads (no padding)
        mb["update"] = 30 * live
        mb["total"] = mb["reduce"] + mb["norm"] + mb["update"]
    return mb


def library_buckets(grs, plan) -> list:
    """The bucket geometry of a libgrs plan (grs_bucket_info per bucket)."""
    nb = grs.grs_plan_query(plan)["n_buckets"]
    return [grs.grs_bucket_info(plan, b) for b in range(nb)]


def oracle_buckets(op) -> list:
    """The same geometry from the oracle's own plan (CPU legs only)."""
    out = []
    for b in range(op.n_buckets):
        tag = int(op.b_tag[b])
        ge = op.world if tag in (0, 1) else (op.dp if tag == 2 else 1)
        out.append({"tag": tag, "copies": op.copies(b), "padded": int(op.b_padded[b]),
                    "used": int(op.b_used[b]), "group_size": ge})
    return out


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.time(), line.strip()))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def mark(self, name):
        self.marks.append((name, time.time()))

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        t0 = dict(self.marks).get("load_start", 0)
        t1 = dict(self.marks).get("load_end", time.time())
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- ranks
def max_over_ranks(x: float, device="cpu") -> float:
    """The largest value over all ranks of the process group (the job's time
    is its slowest replica's); identity without a group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ms_per_step_max: float, world_size: int) -> float:
    """Whole-job ms per update: every rank is an independent replica doing one
    update per step, so N ranks finish N updates in the slowest rank's step."""
    return ms_per_step_max / world_size


# --------------------------------------------------------------------------- GPU arm
def bench_workload(args):
    """The workload named on the command line, with --micro overriding its
    number of microbatches (the name then says so)."""
    import dataclasses
    cid = args.workload if args.workload is not None else (1 if args.blocks else HEADLINE)
    w = workloads.get(cid, args.blocks, getattr(args, "layers", 0))
    if getattr(args, "micro", 0) and args.micro != w.n_micro:
        w = dataclasses.replace(w, n_micro=args.micro, name=f"{w.name}-{args.micro}mb")
    return w


# Variants of the update (the pages' validation list): the same workload with
# fp32 rank gradients; with tensors that have no gradient this step; with
# frozen tensors; or with a trailing accumulation window of fewer
# microbatches.  The patterns are fixed and stated in the JSON line.
VARIANTS = ("plain", "fp32-grads", "unused", "frozen")


def unused_pattern(n_tensors: int) -> list:
    """Tensors without a gradient this step: every 7th, starting at index 3."""
    return [0 if i % 7 == 3 else 1 for i in range(n_tensors)]


def frozen_pattern(n_tensors: int) -> list:
    """Frozen tensors: the first quarter in model order (the lowest layers)."""
    return [1 if i < n_tensors // 4 else 0 for i in range(n_tensors)]


class GpuUpdate:
    """All device buffers of one workload and the calls of one update."""

    def __init__(self, w: workloads.Workload, device, variant: str = "plain", window: int = 0,
                 graph: bool = False, small: bool = False):
        import torch
        from gradient_reduction_sharded_gb300 import grs
        self.torch, self.grs, self.w, self.dev = torch, grs, w, device
        self.variant = variant
        self.n_micro = window if window > 0 else w.n_micro
        if self.n_micro > w.n_micro:
            raise ValueError(f"window {self.n_micro} > the workload's {w.n_micro} microbatches")
        n = len(w.numels)
        self.tensor_flags = frozen_pattern(n) if variant == "frozen" else None
        self.grad_bytes = 4 if variant == "fp32-grads" else 2
        flags = grs.GRS_PLAN_FP32_GRADS if variant == "fp32-grads" else 0
        self.plan = grs.grs_plan_create_ex(w.numels, w.owners, self.tensor_flags, w.world, w.tp,
                                           w.dp_replicate, w.dp_shard, w.bucket_bytes, flags)
        self.info = grs.grs_plan_query(self.plan)
        self.buckets = library_buckets(grs, self.plan)
        nrp, nsp = self.info["n_rank_pad"], self.info["n_state_pad"]
        gen = workloads.normal_f32 if variant == "fp32-grads" else workloads.normal_bf16
        self.grads = [[gen(nrp, w.grad_std, workloads.grad_seed(w.cid, j, k), device=device)
                       for k in range(w.world)] for j in range(self.n_micro)]
        self.ptrs = [[t.data_ptr() for t in mb] for mb in self.grads]
        # the same pointers as C arrays, built once (no per-call conversion)
        self.ptr_arrays = [grs.pointer_array(p) for p in self.ptrs]
        self.all_ptrs = grs.pointer_array([p for mb in self.ptrs for p in mb])
        self.acc = torch.empty(nsp, dtype=torch.float32, device=device)
        self.master = workloads.normal_f32(nsp, w.master_std, workloads.master_seed(w.cid),
                                           device=device)
        self.m = torch.zeros(nsp, dtype=torch.float32, device=device)
        self.v = torch.zeros(nsp, dtype=torch.float32, device=device)
        self.params = torch.empty(nsp, dtype=torch.int16, device=device)
        self.ws = torch.zeros(self.info["workspace_bytes"] // 4 + 4, dtype=torch.float32,
                              device=device)
        self.norm = torch.zeros(1, dtype=torch.float64, device=device)
        self.stream = torch.cuda.current_stream(device).cuda_stream
        self.step_no = 0
        self.used = None
        if variant == "unused":
            self.used_list = unused_pattern(n)
            self.used = torch.tensor(self.used_list, dtype=torch.uint8, device=device)
            self.tensor_steps = torch.zeros(n, dtype=torch.int32, device=device)
        # A CUDA graph replays the launches it captured, host arguments
        # included, so the step count must live on the device: the captured
        # update is the per-tensor-step AdamW with every tensor marked as
        # having a gradient (bit-identical to the plain update), after the
        # plain reduction and norm.
        self.graph = None
        self.graphed = graph
        # One launch for the whole update (grs_update_small): plain updates of
        # plans within its tile and buffer limits only.
        self.small = small
        if small and (variant != "plain" or graph):
            raise ValueError("--small runs the plain eager update only")
        if graph:
            if variant != "plain":
                raise ValueError("--graph runs the plain update only")
            self.all_used = torch.ones(n, dtype=torch.uint8, device=device)
            self.tensor_steps = torch.zeros(n, dtype=torch.int32, device=device)
        # kernels per step: one reduction per microbatch, the norm finish and the
        # update; the masked path adds its norm pass and the per-tensor factors
        self.launches_per_step = self.n_micro + (4 if self.used is not None else 3 if graph else 2)
        if small:
            self.launches_per_step = 1

    def algorithmic_bytes(self) -> dict:
        """Per-kernel algorithmic bytes of one update of this variant."""
        idle, idle_rows = None, None
        if self.used is not None:
            idle = sum(n for n, u in zip(self.w.numels, self.used_list) if not u)
            idle_rows = [0] * len(self.buckets)
            for i, u in enumerate(self.used_list):
                if not u:
                    ti = self.grs.grs_tensor_info(self.plan, i)
                    if ti["bucket"] >= 0:
                        idle_rows[ti["bucket"]] += ti["per_rank"]
        return variant_bytes(self.buckets, self.n_micro, self.grad_bytes, self.info["n_state_pad"],
                             self.info["n_unique"], idle, idle_rows)

    def reduce(self):
        g = self.grs
        for j in range(self.n_micro):
            if self.used is not None:  # tensors without a gradient are not reduced
                g.grs_reduce_all_masked(self.plan, self.ptr_arrays[j], self.acc.data_ptr(), int(j > 0),
                                        int(j == self.n_micro - 1), self.used.data_ptr(), self.ws.data_ptr(),
                                        self.stream)
            else:
                g.grs_reduce_all(self.plan, self.ptr_arrays[j], self.acc.data_ptr(), int(j > 0),
                                 int(j == self.n_micro - 1), self.ws.data_ptr(), self.stream)

    def norm_sq(self):
        # The last reduction emitted the norm partials (masked ones when a
        # mask is given): only the fixed-order finish runs here.
        self.grs.grs_grad_norm_sq(self.plan, self.acc.data_ptr(), self.n_micro,
                                  self.ws.data_ptr(), 1, self.norm.data_ptr(), self.stream)

    def adamw(self):
        a = self.w.adamw
        self.step_no += 1
        hp = self.grs.make_adamw(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm,
                                 self.step_no, self.n_micro)
        if self.used is not None or self.graphed:
            mask = self.used if self.used is not None else self.all_used
            self.grs.grs_clip_adamw_step_masked(self.plan, hp, self.norm.data_ptr(), self.acc.data_ptr(),
                                                self.master.data_ptr(), self.m.data_ptr(),
                                                self.v.data_ptr(), self.params.data_ptr(),
                                                mask.data_ptr(), self.tensor_steps.data_ptr(),
                                                self.ws.data_ptr(), self.stream)
        else:
            self.grs.grs_clip_adamw_step(self.plan, hp, self.norm.data_ptr(), self.acc.data_ptr(),
                                         self.master.data_ptr(), self.m.data_ptr(), self.v.data_ptr(),
                                         self.params.data_ptr(), self.stream)

    def capture(self):
        """Capture one whole update in a CUDA graph; step() then replays it."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        own = self.stream
        with torch.cuda.stream(side):
            self.stream = side.cuda_stream
            try:
                with torch.cuda.graph(g, stream=side):
                    self.reduce()
                    self.norm_sq()
                    self.adamw()
            finally:
                self.stream = own
        torch.cuda.synchronize(self.dev)
        self.graph = g

    def small_step(self):
        a = self.w.adamw
        self.step_no += 1
        hp = self.grs.make_adamw(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm,
                                 self.step_no, self.n_micro)
        self.grs.grs_update_small(self.plan, hp, self.all_ptrs,
                                  self.acc.data_ptr(), self.master.data_ptr(), self.m.data_ptr(),
                                  self.v.data_ptr(), self.params.data_ptr(), self.norm.data_ptr(),
                                  self.stream)

    def step(self):
        if self.graph is not None:
            self.graph.replay()
            return
        if self.small:
            self.small_step()
            return
        self.reduce()
        self.norm_sq()
        self.adamw()

    def close(self):
        self.torch.cuda.synchronize(self.dev)
        self.grs.grs_plan_destroy(self.plan)


# The headline workload when none is named: the largest plan that fits one
# GPU (Llama-3.2-3B-shaped, 3.2B parameters, 134.9 GB of mandatory traffic
# per update); the other large plans are measured in the same run and
# reported beside it.
HEADLINE = 4
ALSO_MEASURED = (1, 2, 3)
# Nominal GB300 HBM3e bandwidth, for a second fraction next to the one
# against the measured copy peak (roofline.frac).
NOMINAL_HBM_GBS = 7900.0


def load_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def measure(u: "GpuUpdate", args, world_size: int, device, gpu_index: int) -> dict:
    """Time one workload's update: W warm-up steps, a soak, exactly K steps
    between barriers (max over ranks), then K more steps with CUDA events
    between the kernels for the per-kernel roofline; SM clocks sampled over
    both regions."""
    import torch
    w = u.w
    mb = u.algorithmic_bytes()
    clocks = ClockSampler(gpu_index)
    clocks.start()
    dist = None
    if world_size > 1:
        import torch.distributed as dist
    # warm-up: the first step initialises the moments (timing sees a warm state)
    clocks.mark("load_start")
    for _ in range(args.warmup):
        u.step()
    torch.cuda.synchronize()
    if args.graph:
        u.capture()  # later steps replay the captured update
    # soak so that the clock samples see the steady state (untimed)
    t_soak = time.time()
    while time.time() - t_soak < args.soak:
        for _ in range(10):
            u.step()
        torch.cuda.synchronize()
    K = args.steps
    # Inputs that fit in L2 would be timed from the cache: then L2 is flushed
    # before every step (a write of twice its size, outside the events) and
    # each step is timed on its own.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or (129 << 20))
    flush = u.n_micro * w.world * u.info["n_rank_pad"] * u.grad_bytes <= l2_bytes
    scrub = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=device) if flush else None

    def flush_l2():
        if scrub is not None:
            scrub.fill_(0.0)

    # Timed region: exactly K steps, back to back, no events in between
    # (one event pair per step when L2 is flushed between steps).
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if flush:
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for a_, b_ in pairs:
            flush_l2()
            a_.record()
            u.step()
            b_.record()
        torch.cuda.synchronize()
        total_ms = sum(a_.elapsed_time(b_) for a_, b_ in pairs)
    else:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record()
        for _ in range(K):
            u.step()
        t_end.record()
        torch.cuda.synchronize()
        total_ms = t_start.elapsed_time(t_end)
    if dist is not None:
        dist.barrier()
    ms_step = max_over_ranks(total_ms / K, device)
    # Per-kernel durations for the roofline: a second region of K steps with
    # CUDA events between the kernels on the launching stream (the events
    # themselves cost a few microseconds per step, so they stay out of the
    # headline region).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        flush_l2()
        ev[i][0].record()
        if u.small:  # one launch: the whole update lands in the first slot
            u.small_step()
            ev[i][1].record()
            ev[i][2].record()
            ev[i][3].record()
            continue
        u.reduce()
        ev[i][1].record()
        u.norm_sq()
        ev[i][2].record()
        u.adamw()
        ev[i][3].record()
    torch.cuda.synchronize()
    clocks.mark("load_end")
    red_ms = [e[0].elapsed_time(e[1]) for e in ev]
    nrm_ms = [e[1].elapsed_time(e[2]) for e in ev]
    upd_ms = [e[2].elapsed_time(e[3]) for e in ev]
    upd_total = sorted(e[0].elapsed_time(e[3]) for e in ev)
    clk = clocks.stop()
    del scrub

    peaks = load_peaks()
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    M = u.n_micro
    masked = u.used is not None
    kern = {
        "reduce": {"ms": statistics.mean(red_ms), "ms_median": statistics.median(red_ms),
                   "bytes": mb["reduce"] / M, "launches_per_step": M},
        "update": {"ms": statistics.mean(upd_ms), "ms_median": statistics.median(upd_ms),
                   "bytes": mb["update"], "launches_per_step": 2 if masked else 1},
        "norm": {"ms": statistics.mean(nrm_ms), "ms_median": statistics.median(nrm_ms),
                 "bytes": None, "launches_per_step": 1},
    }
    # reduce: average per launch over the microbatches of a step
    kern["reduce"]["ms_per_launch"] = kern["reduce"]["ms"] / M
    kern["update"]["ms_per_launch"] = kern["update"]["ms"]
    kern["norm"]["ms_per_launch"] = kern["norm"]["ms"]
    if u.small:
        kern = {"update_small": {"ms": statistics.mean(red_ms), "ms_median": statistics.median(red_ms),
                                 "bytes": mb["total"], "launches_per_step": 1, "ms_per_launch":
                                 statistics.mean(red_ms),
                                 "note": "reduction of every microbatch, norm, clip + AdamW in one cluster launch"}}
    dom = max(kern, key=lambda k: kern[k]["ms"] if kern[k]["bytes"] else -1.0)
    dk = kern[dom]
    achieved = dk["bytes"] / (dk["ms_per_launch"] * 1e-3) / 1e9
    traffic = load_traffic(dom, w, u.variant)
    if masked:
        kern["update"]["note"] = "per-tensor factors kernel + masked update"
        kern["reduce"]["note"] = "masked reduction (masked norm partials fused into the last microbatch)"
    step_gbs = mb["total"] / (ms_step * 1e-3) / 1e9
    return {
        "ms_per_step": ms_step, "flush": flush, "mb": mb,
        "achieved_gbs_total": step_gbs,
        "step_frac": step_gbs / hbm_peak,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": dk["bytes"],
                     "nominal": {"peak": NOMINAL_HBM_GBS, "frac": achieved / NOMINAL_HBM_GBS,
                                 "source": "nominal GB300 HBM3e bandwidth (7.9 TB/s)"},
                     "frac_basis": "frac is against the measured copy peak (peak); nominal.frac against "
                                   "the nominal HBM bandwidth"},
        "kernels": kern,
        "per_update_ms": {"median": statistics.median(upd_total), "min": upd_total[0],
                          "max": upd_total[-1],
                          "note": "second region, one update per event pair (events between kernels add a few us)"},
        "clocks": clk,
    }


def gpu_index_of(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
    return int(vis) if vis.isdigit() else local_rank


def run_gpu(args, rank, world_size, local_rank):
    import torch
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    gpu_index = gpu_index_of(local_rank)
    w = bench_workload(args)
    u = GpuUpdate(w, device, args.variant, args.window, args.graph, args.small)
    plain = args.variant == "plain" and u.n_micro == w.n_micro and not args.graph and not args.small
    r = measure(u, args, world_size, device, gpu_index)
    mb, ms_step, flush = r["mb"], r["ms_per_step"], r["flush"]
    K = args.steps

    # The gather and the end-to-end path run on the plain update only.
    # ---------------------------------------------------------------- gather
    gather = run_gather(u, args, torch) if plain else None
    if gather is not None and flush:
        gather["l2"] = "parameters fit in L2: back-to-back gathers read them from the cache"
    accumulate = run_accumulate(u, args, torch) if plain else None

    # ---------------------------------------------------------------- e2e
    e2e = None
    if not args.no_e2e and plain:
        need = e2e_host_bytes(u)
        ranks_here = int(os.environ.get("LOCAL_WORLD_SIZE", str(world_size)))
        avail = host_available_bytes()
        if avail is None or need * ranks_here <= 0.6 * avail:
            e2e = run_e2e(u, args, torch)
        else:
            # Every rank on this host would pin its own copy of the gradients:
            # the 67M plan stands in, and the line says so.
            w1 = workloads.get(1)
            u1 = GpuUpdate(w1, device)
            u1.step()
            e2e = run_e2e(u1, args, torch)
            e2e["workload"] = w1.name
            e2e["why"] = (f"{need * ranks_here / 1e9:.0f} GB of pinned host memory for {ranks_here} ranks of "
                          f"{w.name} exceeds 60% of the {avail / 1e9:.0f} GB available")
            u1.close()
            del u1

    status = u.grs.grs_check_device_errors(u.plan, u.stream)
    u.close()

    result = {
        "metric": METRIC, "value": job_value(ms_step, world_size), "unit": UNIT, "n_gpus": world_size,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": arm_config(w, u, world_size, flush),
        "achieved_gbs_total": r["achieved_gbs_total"] if world_size == 1
        else mb["total"] / (ms_step * 1e-3) / 1e9,
        "roofline": r["roofline"],
        "kernels": r["kernels"],
        "e2e": e2e,
        "gather": gather,
        "accumulate": accumulate,
        "gpu_launches": u.launches_per_step * K,
        "kernel_timing": "second region of K steps with CUDA events between the kernels",
        "per_update_ms": r["per_update_ms"],
        "clocks": r["clocks"],
        "device_status": status,
    }
    if plain and w.cid in PAGES_CONTEXT and not (args.layers or args.blocks or args.micro or args.window):
        result["pages_context"] = PAGES_CONTEXT[w.cid]
    if rank == 0 and world_size == 1 and not args.no_cpu_baseline:
        if plain:
            result["cpu_baseline"] = cpu_baseline(w, mb, args, u)
        else:
            result["cpu_baseline"] = cpu_baseline_variant(w, u, mb, args)
    del u
    torch.cuda.empty_cache()
    # The other large plans, after the headline (which runs first, in a
    # fresh process), one after another, each freed before the next (only
    # when the headline is the default plain update).
    others = {}
    if args.workload is None and args.variant == "plain" and not (args.graph or args.small or args.window
                                                                  or args.micro or args.blocks or args.layers):
        for cid in ALSO_MEASURED:
            wo = workloads.get(cid)
            uo = GpuUpdate(wo, device)
            r = measure(uo, args, world_size, device, gpu_index)
            st = uo.grs.grs_check_device_errors(uo.plan, uo.stream)
            cfg = arm_config(wo, uo, world_size, r["flush"])
            uo.close()
            del uo
            torch.cuda.empty_cache()
            others[wo.name] = {
                "ms_per_update": job_value(r["ms_per_step"], world_size),
                "ms_per_step": r["ms_per_step"], "mandatory_bytes": r["mb"]["total"],
                "gbs": r["achieved_gbs_total"], "step_frac": r["step_frac"],
                "roofline": {k: r["roofline"][k] for k in ("kernel", "achieved", "peak", "frac", "traffic", "nominal")
                             if k in r["roofline"]},
                "kernels": {k: {"ms_per_launch": v["ms_per_launch"], "launches_per_step": v["launches_per_step"]}
                            for k, v in r["kernels"].items()},
                "config": cfg,
                "clocks": r["clocks"], "device_status": st, "steps": args.steps}
            if cid in PAGES_CONTEXT:
                others[wo.name]["pages_context"] = PAGES_CONTEXT[cid]
    if others:
        result["configs"] = others
    return result


# The one timing of this path that the sources print: a synthetic
# 67M-parameter "draft" benchmark ("refactor(distributed): establish shared
# native TP replica ownership", Preserved prototype and evidence), two
# variants whose names and hardware are not given.  Reported beside the
# 67M plan as context only.
PAGES_CONTEXT = {1: {"ms_per_update": [3.255, 2.624],
                     "note": "the sources' synthetic 67M draft benchmark; hardware, rank count and which "
                             "figure is which variant not stated: context, not a target"}}


def arm_config(w, u, world_size: int, flush: bool) -> dict:
    """The JSON line's config (workload_config) for the update `u` runs."""
    return workload_config(w, u.grad_bytes, world_size, flush, variant_config(u))


def variant_config(u: GpuUpdate) -> dict:
    """The variant's keys for the JSON line's config (none for the plain update)."""
    out = {}
    if u.variant != "plain":
        out["variant"] = u.variant
    if u.graphed:
        out["cuda_graph"] = "whole update replayed from one capture (device step counts)"
    if u.small:
        out["single_launch"] = "grs_update_small: one thread-block cluster for the whole update"
    if u.n_micro != u.w.n_micro:
        out["window"] = {"microbatches": u.n_micro, "of": u.w.n_micro}
        out["microbatches"] = u.n_micro
    if u.variant == "unused":
        n_off = u.used_list.count(0)
        out["unused"] = {"pattern": "every 7th tensor from index 3 has no gradient",
                         "tensors": n_off,
                         "elements": sum(n for n, k in zip(u.w.numels, u.used_list) if not k)}
    if u.variant == "frozen":
        out["frozen"] = {"pattern": "first quarter of the tensors in model order",
                         "tensors": sum(u.tensor_flags),
                         "elements": sum(n for n, f in zip(u.w.numels, u.tensor_flags) if f)}
        out["params_trained"] = u.info["n_unique"]
    return out


def run_gather(u: GpuUpdate, args, torch):
    """Per-tensor bf16 parameters, two ways, each timed on its own (neither
    is part of the update: parameters can also be used as views of the
    bucket-ordered buffer):
      * grs_gather_params after the update (a separate pass: read + write 2
        bytes per parameter);
      * grs_clip_adamw_step_to_tensors, the update writing each bf16 value
        straight into its tensor (no bucket-ordered copy), against the plain
        update grs_clip_adamw_step in the same loop: its added time is the
        cost of per-tensor output when fused."""
    w = u.w
    outs = [torch.empty(n, dtype=torch.int16, device=u.dev) for n in w.numels]
    ptrs = [t.data_ptr() for t in outs]
    table = torch.tensor(ptrs, dtype=torch.int64, device=u.dev)
    g = u.grs
    for _ in range(3):
        g.grs_gather_params(u.plan, u.params.data_ptr(), ptrs, u.stream)
    torch.cuda.synchronize()

    def timed(fn):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(args.steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / args.steps

    ms = timed(lambda: g.grs_gather_params(u.plan, u.params.data_ptr(), ptrs, u.stream))
    nbytes = 4 * w.n_unique
    a = w.adamw
    hp = g.make_adamw(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, max(1, u.step_no), u.n_micro)

    def plain():
        g.grs_clip_adamw_step(u.plan, hp, u.norm.data_ptr(), u.acc.data_ptr(), u.master.data_ptr(),
                              u.m.data_ptr(), u.v.data_ptr(), u.params.data_ptr(), u.stream)

    def fused():
        g.grs_clip_adamw_step_to_tensors(u.plan, hp, u.norm.data_ptr(), u.acc.data_ptr(), u.master.data_ptr(),
                                         u.m.data_ptr(), u.v.data_ptr(), None, table.data_ptr(), u.stream)

    for _ in range(3):
        plain()
        fused()
    torch.cuda.synchronize()
    ms_plain, ms_fused = [], []
    for _ in range(3):  # interleaved, the best of three loops each
        ms_plain.append(timed(plain))
        ms_fused.append(timed(fused))
    p_ms, f_ms = min(ms_plain), min(ms_fused)
    upd_bytes = 30 * u.info["n_state_pad"]
    del outs, table
    return {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "fused_into_update": {
                "update_ms": p_ms, "update_to_tensors_ms": f_ms, "added_ms": f_ms - p_ms,
                "added_frac_of_separate_gather": (f_ms - p_ms) / ms,
                "update_to_tensors_gbs": upd_bytes / (f_ms * 1e-3) / 1e9,
                "bytes_per_element": 30,
                "note": "grs_clip_adamw_step_to_tensors with no bucket-ordered copy, against "
                        "grs_clip_adamw_step, best of 3 interleaved loops of K calls each"}}


def run_accumulate(u: GpuUpdate, args, torch):
    """grs_accumulate over every bucket (adding a separately reduced fp32
    microbatch into the accumulator), timed on its own: it is not on the
    update's path, where the reduction accumulates in its own epilogue.
    Algorithmic bytes: read acc and the microbatch, write acc, 4 each."""
    mbuf = torch.zeros_like(u.acc)
    nsp = u.info["n_state_pad"]
    offs = [(b, int(d["state_offset"])) for b, d in enumerate(u.buckets)]

    def once():
        for b, off in offs:
            u.grs.grs_accumulate(u.plan, b, u.acc.data_ptr() + 4 * off, mbuf.data_ptr() + 4 * off, u.stream)

    for _ in range(3):
        once()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        once()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.steps
    nbytes = 12 * nsp
    del mbuf
    return {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9, "launches": len(offs)}


def e2e_host_bytes(u: GpuUpdate) -> int:
    """Pinned host bytes run_e2e allocates for `u`: every rank's gradients of
    every microbatch and the bf16 parameters read back."""
    return (u.n_micro * u.w.world * u.info["n_rank_pad"] + u.info["n_state_pad"]) * 2


def host_available_bytes():
    """MemAvailable of this host (Linux), or None when it cannot be read."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def run_e2e(u: GpuUpdate, args, torch):
    """The same update through the public C ABI with host buffers:
    grs_step_from_host copies every step's gradients from pinned host memory
    (bucket by bucket, overlapped with the reductions), runs the update and
    reads the step's results back to the host every step: the bf16
    parameters and the squared global norm (a second figure reads the norm
    alone)."""
    w = u.w
    W, M = w.world, w.n_micro
    n = u.info["n_rank_pad"]
    t0 = time.perf_counter()
    host = [torch.empty(n, dtype=torch.int16, pin_memory=True) for _ in range(M * W)]
    for j in range(M):
        for k in range(W):
            host[j * W + k].copy_(u.grads[j][k].view(torch.int16))
    halves = 2 if M > 1 else 1
    stage = [torch.empty(n, dtype=torch.bfloat16, device=u.dev) for _ in range(halves * W)]
    stage_ptrs = [t.data_ptr() for t in stage] + [stage[0].data_ptr()] * ((2 - halves) * W)
    out_params = torch.empty(u.params.numel(), dtype=torch.int16, pin_memory=True)
    out_norm = torch.empty(1, dtype=torch.float64, pin_memory=True)
    t_setup = time.perf_counter() - t0  # pinned host buffers, filled from the device
    h2d = 0
    for d in u.buckets:  # ALREADY_REDUCED buckets copy rank 0's rows only
        nread = 1 if int(d["tag"]) == 3 else W
        h2d += M * nread * int(d["padded"]) * 2
    d2h = out_params.numel() * 2 + 8
    steps = max(3, min(args.steps, 20))  # pipeline fill and drain (~1 ms) spread over the steps
    a = w.adamw

    def one(read_params: bool):
        u.step_no += 1
        hp = u.grs.make_adamw(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, u.step_no, M)
        u.grs.grs_step_from_host(u.plan, hp, [t.data_ptr() for t in host], stage_ptrs,
                                 u.acc.data_ptr(), u.master.data_ptr(), u.m.data_ptr(), u.v.data_ptr(),
                                 u.params.data_ptr(), u.ws.data_ptr(), u.norm.data_ptr(),
                                 out_params.data_ptr() if read_params else None, out_norm.data_ptr(), u.stream)

    def timed(read_params: bool):
        """Mean ms per step over the bracketed loop, and each step's interval
        (event after each call on the same stream; the first interval holds
        the pipeline fill, as the first step's copies overlap nothing)."""
        one(read_params)
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record()
        for i in range(steps):
            one(read_params)
            evs[i + 1].record()
        torch.cuda.synchronize()
        per = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(steps))
        return evs[0].elapsed_time(evs[-1]) / steps, {"median": per[len(per) // 2], "min": per[0],
                                                      "max": per[-1]}

    # The host link on this machine, for scale: one pinned 1 GiB copy each way
    # (host-to-device also before the timed loops; the host link is shared
    # and its rate changes over seconds).
    nb = min(n, 1 << 29)
    hsrc, dbuf = host[0][:nb], stage[0].view(torch.int16)[:nb]

    def copy_ms(fn):
        fn()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(3):
            fn()
        s1.record()
        torch.cuda.synchronize()
        return s0.elapsed_time(s1) / 3

    h2d_before = 2 * nb / (copy_ms(lambda: dbuf.copy_(hsrc, non_blocking=True)) * 1e-3) / 1e9
    # The step's result read back every step: the updated bf16 parameters
    # and the squared global norm; as a second figure, the norm alone.
    ms_params, per_params = timed(True)
    ms, per_norm = timed(False)
    link = {"h2d_gbs": 2 * nb / (copy_ms(lambda: dbuf.copy_(hsrc, non_blocking=True)) * 1e-3) / 1e9,
            "d2h_gbs": 2 * nb / (copy_ms(lambda: hsrc.copy_(dbuf, non_blocking=True)) * 1e-3) / 1e9,
            "h2d_gbs_before": h2d_before,
            "bytes": 2 * nb, "note": "one pinned buffer copied each way after the timed loops (host-to-device "
                                     "also before them), cudaMemcpyAsync via torch; link_bound_ms adds the two "
                                     "directions (no overlap)"}
    del stage
    return {"value": ms_params, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_gbs": h2d / (ms_params * 1e-3) / 1e9, "steps": steps,
            "per_step_ms": per_params,
            "setup_s": t_setup,
            "path": "grs_step_from_host: pinned host gradients, per-bucket H2D overlapped with the "
                    "reductions; the bf16 parameters and the squared global norm read back every step",
            "norm_read_back_only": {"value": ms, "unit": UNIT, "d2h_bytes_per_step": 8,
                                    "h2d_gbs": h2d / (ms * 1e-3) / 1e9, "per_step_ms": per_norm},
            "link": link,
            "link_bound_ms": (h2d / link["h2d_gbs"] + (d2h - 8) / link["d2h_gbs"]) / 1e6
            if link["h2d_gbs"] > 0 and link["d2h_gbs"] > 0 else None}


KERNEL_SOURCES = ("kernels_reduce.cu", "kernels_update.cu", "kernels_masked.cu", "kernels_gather.cu",
                  "device.cuh", "internal.h", "launch.cuh")


def csrc_hash() -> str:
    """Hash of the sources that define the reduce and update kernels, to tell
    whether stored DRAM counters still apply."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gradient_reduction_sharded_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, w, variant: str = "plain"):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    workload was not captured or the kernels changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("csrc_sha256_16") != csrc_hash():
        return None
    key = f"{kernel}:{w.name}" if variant == "plain" else f"{kernel}:{w.name}:{variant}"
    ent = t.get(key)
    return None if ent is None else ent.get("bytes_per_launch")


# --------------------------------------------------------------------------- CPU arm
def _host_inputs(w, n_rank_pad: int, n_micro: int = 0, fp32: bool = False, device=None):
    """The workload's gradients as host arrays (uint16 bf16 bits, or float32
    with fp32=True), generated exactly as the GPU arm generates them (same
    seeds), one buffer per (microbatch, rank)."""
    import torch
    dev = device or ("cuda" if torch.cuda.is_available() else "cpu")
    gen = workloads.normal_f32 if fp32 else workloads.normal_bf16
    out = []
    for j in range(n_micro or w.n_micro):
        row = []
        for k in range(w.world):
            t = gen(n_rank_pad, w.grad_std, workloads.grad_seed(w.cid, j, k), device=dev)
            row.append(t.cpu().numpy() if fp32 else workloads.bf16_bits(t.cpu()))
            del t
        out.append(row)
    return out


def _sampled_host_inputs(w, op, buckets, n_micro: int = 0, fp32: bool = False, device=None):
    """Only the sampled buckets' inputs [M][R][P], generated exactly as the
    GPU arm generates them (whole per-rank buffers from the same seeds, on
    the device when there is one) and sliced, so that host memory holds only
    the sample."""
    import torch
    dev = device or ("cuda" if torch.cuda.is_available() else "cpu")
    gen = workloads.normal_f32 if fp32 else workloads.normal_bf16
    M = n_micro or w.n_micro
    out = {b: np.zeros((M, w.world, int(op.b_padded[b])), np.float32 if fp32 else np.uint16) for b in buckets}
    for j in range(M):
        for k in range(w.world):
            t = gen(op.n_rank_pad, w.grad_std, workloads.grad_seed(w.cid, j, k), device=dev)
            for b in buckets:
                ro, P = int(op.b_rank_off[b]), int(op.b_padded[b])
                sl = t[ro:ro + P].cpu()
                out[b][j, k] = sl.numpy() if fp32 else workloads.bf16_bits(sl)
            del t
    return out


def _host_fetch(op, host, M):
    """Bucket inputs [M][R][P] sliced from whole per-rank host buffers."""
    def fetch(b):
        ro, P = int(op.b_rank_off[b]), int(op.b_padded[b])
        return np.stack([np.stack([h[ro:ro + P] for h in mb]) for mb in host[:M]])
    return fetch


def _device_bucket_inputs(op, grads, buckets, M, fp32):
    """The sampled buckets' inputs [M][R][P] copied once from the GPU arm's own
    device gradients (the same seeded bytes), so that only the sample is held
    on the host."""
    import torch
    out = {}
    for b in buckets:
        ro, P = int(op.b_rank_off[b]), int(op.b_padded[b])
        arr = np.stack([np.stack([g[ro:ro + P].view(torch.float32 if fp32 else torch.int16).cpu().numpy()
                                  for g in mb]) for mb in grads[:M]])
        out[b] = arr if fp32 else arr.view(np.uint16)
    return out


def _oracle_sample(w, op, host, buckets, threads=1, n_micro=0, used=None, master=None):
    """One oracle update restricted to `buckets` (reduce -> norm -> AdamW);
    with threads > 1 the buckets run in parallel (the oracle's C code drops
    the GIL) and the norm is still summed in bucket order.  With `used` (one
    flag per tensor) tensors without a gradient add nothing to the norm and
    are not updated.  `master` (dict bucket -> fp32 [copies * P], or None for
    zeros) is the state the step starts from; the first and second moments
    start at zero (the first step), each in an array of its own."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    a_ = w.adamw
    hp = (a_.lr, a_.beta1, a_.beta2, a_.eps, a_.weight_decay)
    M = n_micro or w.n_micro

    def rows(b):
        """(row, lo, hi): the ranges of bucket b's tensors with a gradient."""
        out = []
        for i in range(len(op.numel)):
            if int(op.t_bucket[i]) == b and used[i]:
                o, n = int(op.t_offset[i]), op.per_rank(i)
                out += [(t, o, o + n) for t in range(op.copies(b))]
        return out

    fetch = host.__getitem__ if isinstance(host, dict) else _host_fetch(op, host, M)

    def red(b):
        P = int(op.b_padded[b])
        g = fetch(b)
        a = oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard, P,
                                 int(op.b_used[b]), g)
        if used is None:
            return a, oracle.norm_sq(a, M)
        ns = 0.0
        for t, lo, hi in rows(b):
            ns += oracle.norm_sq(a[t][lo:hi], M)
        return a, ns

    def state(b, t, lo, hi):
        P = int(op.b_padded[b])
        p0 = (master[b][t * P + lo:t * P + hi] if master is not None
              else np.zeros(hi - lo, np.float32))
        return p0, np.zeros(hi - lo, np.float32), np.zeros(hi - lo, np.float32)

    def upd(args):
        b, a, c = args
        if used is None:
            P = int(op.b_padded[b])
            for t in range(op.copies(b)):
                oracle.adamw(a[t], int(op.b_used[b]), M, c, hp, 1, *state(b, t, 0, P))
            return
        for t, lo, hi in rows(b):
            oracle.adamw(a[t][lo:hi], hi - lo, M, c, hp, 1, *state(b, t, lo, hi))

    with ThreadPoolExecutor(max(1, threads)) as ex:
        parts = list(ex.map(red, buckets))
        s = 0.0
        for _, ns in parts:
            s += ns
        c = oracle.clip_coef(s, w.adamw.max_norm)
        list(ex.map(upd, [(b, a, c) for b, (a, _) in zip(buckets, parts)]))
    return s


def _sample_buckets(op, frac_target=0.35):
    """A bounded sample of the same workload: for every tag the bucket
    closest in size to the median bucket, then buckets in plan order that are
    at most twice the median (no single outsized bucket, such as one holding
    a whole embedding, can dominate a sample), until ~frac_target of the
    state elements are covered."""
    total = op.n_state_pad
    sizes = [op.copies(b) * int(op.b_padded[b]) for b in range(op.n_buckets)]
    med = sorted(sizes)[len(sizes) // 2] if sizes else 0
    chosen, acc = [], 0
    by_tag = {}
    for b in range(op.n_buckets):
        by_tag.setdefault(int(op.b_tag[b]), []).append(b)
    for tag, bs in sorted(by_tag.items()):
        b = min(bs, key=lambda x: (abs(sizes[x] - med), x))
        chosen.append(b)
        acc += sizes[b]
    for b in range(op.n_buckets):
        if acc >= frac_target * total:
            break
        if b not in chosen and sizes[b] <= 2 * med:
            chosen.append(b)
            acc += sizes[b]
    return sorted(chosen)


def _sample_bytes(op, buckets, n_micro, grad_bytes=2):
    """Mandatory bytes of the sampled buckets (the plain update's formula)."""
    geo = oracle_buckets(op)
    return mandatory_bytes([geo[b] for b in buckets], n_micro, grad_bytes)["total"]


def _oracle_plan(w, tensor_flags=None):
    import oracle
    return oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard,
                       w.bucket_bytes, tensor_flags)


def cpu_baseline(w, mb, args, u=None, target_s=10.0):
    """The oracle as it stands, on this host: whole updates of the workload
    (every bucket: reduce -> norm -> AdamW), repeated until about target_s of
    CPU work, one thread; then the same with one thread per core (buckets in
    parallel).  An update that moves more than 8 GB is sampled instead (one
    bucket per tag, scaled to the whole update by mandatory bytes), its
    inputs copied once from the GPU arm's own gradients (`u`), so that host
    memory holds only the sample."""
    if mb["total"] > 8e9 and u is not None:
        return cpu_baseline_variant(w, u, mb, args, target_s)
    op = _oracle_plan(w)
    host = _host_inputs(w, op.n_rank_pad)
    buckets = list(range(op.n_buckets))
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_sample(w, op, host, buckets)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= target_s or reps >= 20:
            break
    ms = dt * 1e3 / reps
    nthr = os.cpu_count() or 1
    t1 = time.perf_counter()
    _oracle_sample(w, op, host, buckets, threads=nthr)
    dtn = time.perf_counter() - t1
    return {"value": ms, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} whole updates of the workload ({op.n_buckets} buckets, "
                      f"{mb['total'] / 1e9:.2f} GB mandatory bytes each), one thread, {dt:.1f} s",
            "gbs": mb["total"] / (ms * 1e-3) / 1e9,
            "all_cores": {"value": dtn * 1e3, "cores": nthr, "gbs": mb["total"] / dtn / 1e9,
                          "note": f"one whole update, {min(nthr, op.n_buckets)} buckets in parallel"}}


def _spread_buckets(op, n):
    """Up to n buckets for a parallel sample: _sample_buckets' one per tag,
    then others of at most twice the median bucket size in plan order (so
    that the threads get comparable work)."""
    chosen = _sample_buckets(op, frac_target=0.0)
    sizes = [op.copies(b) * int(op.b_padded[b]) for b in range(op.n_buckets)]
    med = sorted(sizes)[len(sizes) // 2] if sizes else 0
    for b in range(op.n_buckets):
        if len(chosen) >= n:
            break
        if b not in chosen and sizes[b] <= 2 * med:
            chosen.append(b)
    return sorted(chosen)


def _master_slices(op, master, buckets):
    """Each sampled bucket's rows of an fp32 state array (torch, any device)
    as host arrays."""
    out = {}
    for b in buckets:
        o = int(op.b_state_off[b])
        out[b] = master[o:o + op.copies(b) * int(op.b_padded[b])].cpu().numpy()
    return out


def cpu_baseline_variant(w, u, mb, args, target_s=10.0):
    """The oracle on the update `u` runs (its plan flags, gradient type,
    microbatch window and mask), one thread: whole updates when the update
    moves at most 8 GB, otherwise one bucket per tag scaled to the whole
    update by mandatory bytes; then one thread per core over as many
    buckets, also scaled.  Inputs: the GPU arm's own gradient bytes and
    master state, copied to the host once before the timing."""
    op = _oracle_plan(w, u.tensor_flags)
    M = u.n_micro
    nthr = os.cpu_count() or 1
    whole = mb["total"] <= 8e9
    buckets = list(range(op.n_buckets)) if whole else _sample_buckets(op, frac_target=0.0)
    par = buckets if whole else _spread_buckets(op, nthr)
    host = _device_bucket_inputs(op, u.grads, par, M, u.grad_bytes == 4)
    master = _master_slices(op, u.master, par)
    used = u.used_list if u.used is not None else None
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_sample(w, op, host, buckets, n_micro=M, used=used, master=master)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= target_s or reps >= 20:
            break
    scale = 1.0 if whole else mb["total"] / _sample_bytes(op, buckets, M, u.grad_bytes)
    ms = dt * 1e3 / reps * scale
    t1 = time.perf_counter()
    _oracle_sample(w, op, host, par, threads=nthr, n_micro=M, used=used, master=master)
    dtn = time.perf_counter() - t1
    scale_n = 1.0 if whole else mb["total"] / _sample_bytes(op, par, M, u.grad_bytes)
    msn = dtn * 1e3 * scale_n
    what = (f"{reps} whole updates" if whole else
            f"{reps} updates of buckets {buckets} of {op.n_buckets}, scaled by mandatory bytes")
    return {"value": ms, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{what}, one thread, {dt:.1f} s", "gbs": mb["total"] / (ms * 1e-3) / 1e9,
            "all_cores": {"value": msn, "cores": nthr, "gbs": mb["total"] / (msn * 1e-3) / 1e9,
                          "note": (f"one whole update, {min(nthr, len(par))} buckets in parallel" if whole else
                                   f"one update of {len(par)} buckets in parallel, scaled by mandatory bytes")}}


def workload_config(w, grad_bytes: int, world_size: int, flush: bool, extra=None) -> dict:
    """The JSON line's config, the same for both arms: the workload's
    geometry, gradient type, L2 handling of the GPU timing, parallelism and
    a variant's keys."""
    return dict(w.describe(), grad_dtype="fp32" if grad_bytes == 4 else "bf16",
                l2=("L2 flushed before every step (inputs fit in L2)" if flush
                    else "inputs larger than L2 (no flush)"),
                parallelism=f"replicas{world_size}" if world_size > 1 else "1 GPU, simulated ranks",
                **(extra or {}))


def run_reference(args, rank, world_size):
    """The oracle as the reference arm, on the host cores, rank 0 only, on
    the GPU arm's workload.  One thread per core, buckets in parallel.  A
    step is one whole oracle update when the update moves at most 5 GB of
    mandatory bytes; otherwise a bounded sample of as many buckets as there
    are cores, and the metric (ms per whole update) is the sample's time
    scaled by mandatory bytes.  ms_per_step is the measured time of one
    step as run."""
    import torch
    w = bench_workload(args)
    op = _oracle_plan(w)
    mb = mandatory_bytes(oracle_buckets(op), w.n_micro)
    nthr = os.cpu_count() or 1
    whole = mb["total"] <= 5e9
    buckets = list(range(op.n_buckets)) if whole else _spread_buckets(op, nthr)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    host = _sampled_host_inputs(w, op, buckets, device=dev)
    master_full = workloads.normal_f32(op.n_state_pad, w.master_std, workloads.master_seed(w.cid), device=dev)
    master = _master_slices(op, master_full, buckets)
    del master_full
    sb = _sample_bytes(op, buckets, w.n_micro)
    for _ in range(args.warmup):
        _oracle_sample(w, op, host, buckets, threads=nthr, master=master)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_sample(w, op, host, buckets, threads=nthr, master=master)
    dt = (time.perf_counter() - t0) / args.steps
    ms_step = dt * 1e3
    ms = ms_step * mb["total"] / sb
    l2 = 129 << 20
    flush = w.n_micro * w.world * op.n_rank_pad * 2 <= l2
    if whole:
        sample = (f"each step: one whole oracle update ({op.n_buckets} buckets, {mb['total'] / 1e9:.2f} GB "
                  f"mandatory bytes), {nthr} threads")
    else:
        sample = (f"each step: oracle update of {len(buckets)} of {op.n_buckets} buckets "
                  f"({sb / 1e9:.2f} of {mb['total'] / 1e9:.2f} GB mandatory bytes), {nthr} threads; "
                  f"value = step time x {mb['total'] / sb:.2f} (bytes of the whole update / bytes of the sample)")
    return {"metric": METRIC, "value": ms, "unit": UNIT, "n_gpus": world_size, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(w, 2, world_size, flush),
            "value_basis": "measured whole updates" if whole else "sampled buckets scaled by mandatory bytes",
            "where": "the oracle (plain C, fp64) on the host cores; inputs in host memory",
            "cpu_baseline": {"value": ms, "unit": UNIT, "cores": nthr, "kind": "oracle", "sample": sample},
            "e2e": {"value": ms, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def reshard_geometry(w):
    """The reader geometry of the reshard measurement: HSDP -> FSDP (every DP
    rank a shard) when the writer has replicas, else two replicas."""
    dr, ds = w.dp_replicate, w.dp_shard
    if dr > 1:
        return w.tp, 1, dr * ds
    if ds % 2 == 0:
        return w.tp, 2, ds // 2
    return w.tp, dr, ds


def run_checkpoint(args):
    """Checkpoint restore with reshard (a separate measurement, not the bench
    line): master, m and v of the workload's plan moved to the canonical
    logical order with the writer's plan (grs_state_to_logical) and into
    another geometry's bucket layout (grs_state_from_logical).  Algorithmic
    bytes per array: read + write 4 bytes per logical element for each
    kernel (the reader also writes its padding zeros).  The end-to-end leg
    saves the three arrays to shard files and loads them into the reader's
    plan through checkpoint.save / checkpoint.load (host file I/O)."""
    import shutil
    import tempfile

    import torch

    from gradient_reduction_sharded_gb300 import checkpoint as ck
    from gradient_reduction_sharded_gb300 import grs
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = bench_workload(args)
    tp, dr, ds = reshard_geometry(w)
    spec_w = ck.PlanSpec(list(w.numels), list(w.owners), None, w.world, w.tp, w.dp_replicate,
                         w.dp_shard, w.bucket_bytes)
    spec_r = ck.PlanSpec(list(w.numels), list(w.owners), None, w.world, tp, dr, ds, w.bucket_bytes)
    pw, pr = spec_w.create(), spec_r.create()
    iw, ir = grs.grs_plan_query(pw), grs.grs_plan_query(pr)
    N = iw["n_unique"]
    names = ("master", "exp_avg", "exp_avg_sq")
    src = {nm: workloads.normal_f32(iw["n_state_pad"], 0.02, 7_919 + w.cid + i, device=device)
           for i, nm in enumerate(names)}
    dst = {nm: torch.empty(ir["n_state_pad"], dtype=torch.float32, device=device) for nm in names}
    logical = torch.empty(max(1, N), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device).cuda_stream
    clocks = ClockSampler(0)
    clocks.start()

    def one(ev=None):
        for nm in names:
            if ev is not None:
                ev[0].record()
            grs.grs_state_to_logical(pw, src[nm].data_ptr(), logical.data_ptr(), stream)
            if ev is not None:
                ev[1].record()
            grs.grs_state_from_logical(pr, logical.data_ptr(), dst[nm].data_ptr(), stream)
            if ev is not None:
                ev[2].record()
                ev = ev[3:]

    clocks.mark("load_start")
    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(K):
        one()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / K
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(K)]
    for i in range(K):
        one(evs[i])
    torch.cuda.synchronize()
    clocks.mark("load_end")
    clk = clocks.stop()
    to_ms = [e[3 * a].elapsed_time(e[3 * a + 1]) for e in evs for a in range(3)]
    from_ms = [e[3 * a + 1].elapsed_time(e[3 * a + 2]) for e in evs for a in range(3)]
    b_to = 8 * N
    b_from = 8 * N + 4 * (ir["n_state_pad"] - N)
    kern = {"state_to_logical": {"ms_per_launch": statistics.median(to_ms), "bytes": b_to,
                                 "launches_per_step": 3},
            "state_from_logical": {"ms_per_launch": statistics.median(from_ms), "bytes": b_from,
                                   "launches_per_step": 3,
                                   "note": "plus one padding-zero launch per call"}}
    dom = max(kern, key=lambda k: kern[k]["ms_per_launch"])
    achieved = kern[dom]["bytes"] / (kern[dom]["ms_per_launch"] * 1e-3) / 1e9
    # correctness of what was timed: the reader's logical order equals the writer's
    back = torch.empty_like(logical)
    for nm in names:
        grs.grs_state_to_logical(pr, dst[nm].data_ptr(), back.data_ptr(), stream)
        grs.grs_state_to_logical(pw, src[nm].data_ptr(), logical.data_ptr(), stream)
        torch.cuda.synchronize()
        if not torch.equal(back, logical):
            raise RuntimeError(f"reshard of {nm} does not round-trip")
    # end to end through the checkpoint module: files on local disk
    tmp = tempfile.mkdtemp(prefix="grs-bench-ckpt-")
    try:
        d = os.path.join(tmp, "ckpt")
        torch.cuda.synchronize()
        s0 = time.perf_counter()
        ck.save(d, pw, spec_w, src, {"step": 1})
        s1 = time.perf_counter()
        ck.load(d, pr, dst)
        s2 = time.perf_counter()
        file_bytes = sum(os.path.getsize(os.path.join(d, f)) for f in os.listdir(d))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    status = grs.grs_check_device_errors(pr, stream)
    grs.grs_plan_destroy(pw)
    grs.grs_plan_destroy(pr)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    res = {"metric": "ms per reshard restore of master, m and v (state -> logical -> other layout)",
           "value": ms, "unit": "ms/restore", "n_gpus": 1, "steps": K, "warmup": args.warmup,
           "ms_per_step": ms, "higher_is_better": False, "dtype": "f32", "data": "synthetic",
           "config": {"workload": w.name, "params": N,
                      "writer": {"tp": w.tp, "dp_replicate": w.dp_replicate, "dp_shard": w.dp_shard},
                      "reader": {"tp": tp, "dp_replicate": dr, "dp_shard": ds},
                      "arrays": len(names), "l2": "arrays larger than L2 (no flush)"},
           "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak,
                        "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": load_traffic(dom, w, "checkpoint"),
                        "peak_source": "measured" if "hbm_gbs" in peaks else "fallback",
                        "algorithmic_bytes_per_launch": kern[dom]["bytes"]},
           "kernels": kern,
           "gpu_launches": 9 * K,
           "e2e": {"save_ms": (s1 - s0) * 1e3, "load_ms": (s2 - s1) * 1e3, "file_bytes": file_bytes,
                   "d2h_bytes": 4 * iw["n_state_pad"] * len(names),
                   "h2d_bytes": 4 * iw["n_state_pad"] * len(names),
                   "path": "checkpoint.save (D2H, shard files, digests, manifest, _SUCCESS) then "
                           "checkpoint.load into the reader's plan (read, verify, H2D, two layout kernels)"},
           "clocks": clk, "device_status": status}
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_reshard(w, spec_r, src, names)
    return res


def cpu_baseline_reshard(w, spec_r, src, names, target_s=10.0):
    """The oracle's layout functions on the same arrays, one thread."""
    import oracle
    opw = _oracle_plan(w)
    opr = oracle.plan(spec_r.numels, spec_r.owners, spec_r.world, spec_r.tp, spec_r.dp_replicate,
                      spec_r.dp_shard, spec_r.bucket_bytes)
    host = {nm: src[nm].cpu().numpy() for nm in names}
    reps, t0 = 0, time.perf_counter()
    while True:
        for nm in names:
            oracle.from_logical(opr, oracle.to_logical(opw, host[nm]))
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= target_s or reps >= 20:
            break
    return {"value": dt * 1e3 / reps, "unit": "ms/restore", "cores": 1, "kind": "oracle",
            "sample": f"{reps} whole restores of the {len(names)} arrays, one thread, {dt:.1f} s"}


def run_overlap(args):
    """Reduction overlapped with a simulated backward pass (a separate
    measurement, not the bench line).  The backward is one bf16 GEMM per
    bucket (tensor-core bound, --gemm n: n x n x n), in reverse bucket order
    on its own stream, recording an event when each bucket's gradients are
    'ready'; the reductions run on a side stream as soon as their events
    fire, with the grid capped at --max-ctas CTAs, then the norm finish and
    clip + AdamW.  Compared with the same work serialized (all GEMMs, then
    the grouped reduction and the update)."""
    import torch
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = bench_workload(args)
    u = GpuUpdate(w, device)
    g = u.grs
    nb = u.info["n_buckets"]
    n = args.gemm
    A = torch.randn(n, n, device=device, dtype=torch.bfloat16)
    B = torch.randn(n, n, device=device, dtype=torch.bfloat16)
    C = torch.empty(n, n, device=device, dtype=torch.bfloat16)
    bk = [g.grs_bucket_info(u.plan, b) for b in range(nb)]
    main = torch.cuda.current_stream(device)
    back = torch.cuda.Stream(device)
    side = torch.cuda.Stream(device)
    a = w.adamw

    def hp():
        u.step_no += 1
        return g.make_adamw(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, u.step_no, w.n_micro)

    def backward_only():
        for b in reversed(range(nb)):
            torch.matmul(A, B, out=C)

    def serialized():
        for _ in range(w.n_micro):
            backward_only()
        u.step()

    def overlapped():
        start = torch.cuda.Event()
        start.record(main)
        back.wait_event(start)
        side.wait_event(start)
        for j in range(w.n_micro):
            for b in reversed(range(nb)):
                ev = torch.cuda.Event()
                with torch.cuda.stream(back):
                    torch.matmul(A, B, out=C)
                    ev.record(back)
                d = bk[b]
                rp = [p + 2 * d["rank_offset"] for p in u.ptrs[j]]
                g.grs_reduce_bucket_ex(u.plan, b, rp, u.acc.data_ptr() + 4 * d["state_offset"], int(j > 0),
                                       int(j == w.n_micro - 1), u.ws.data_ptr(), args.max_ctas,
                                       ev.cuda_event, side.cuda_stream)
        g.grs_grad_norm_sq(u.plan, u.acc.data_ptr(), w.n_micro, u.ws.data_ptr(), 1, u.norm.data_ptr(),
                           side.cuda_stream)
        g.grs_clip_adamw_step(u.plan, hp(), u.norm.data_ptr(), u.acc.data_ptr(), u.master.data_ptr(),
                              u.m.data_ptr(), u.v.data_ptr(), u.params.data_ptr(), side.cuda_stream)
        done = torch.cuda.Event()
        done.record(side)
        main.wait_event(done)
        done2 = torch.cuda.Event()
        done2.record(back)
        main.wait_event(done2)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(main)
        for _ in range(args.steps):
            fn()
        s1.record(main)
        torch.cuda.synchronize()
        return s0.elapsed_time(s1) / args.steps

    t_back = timed(lambda: [backward_only() for _ in range(w.n_micro)])
    t_ser = timed(serialized)
    t_ovl = timed(overlapped)
    status = g.grs_check_device_errors(u.plan, u.stream)
    u.close()
    return {"metric": "ms per step: simulated backward (bf16 GEMM per bucket) + reduce+clip+AdamW",
            "unit": "ms/step", "workload": w.name, "gemm": n, "buckets": nb, "microbatches": w.n_micro,
            "max_ctas": args.max_ctas, "backward_only": t_back, "serialized": t_ser, "overlapped": t_ovl,
            "hidden_fraction_of_update": (t_ser - t_ovl) / max(1e-9, t_ser - t_back),
            "device_status": status}


def rank_launch_cmd(n_gpus: int, argv, port: int) -> list:
    """The torchrun command that runs this bench as n_gpus ranks on one node
    (one process per GPU, rendezvous on 127.0.0.1) with the same arguments."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n_gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=None, choices=workloads.ALL_IDS,
                    help="time this workload only (default: the 3.2B plan as the headline, "
                         "the 67M, 1.1B and MoE plans measured beside it)")
    ap.add_argument("--blocks", type=int, default=0,
                    help="shrink workload 1 to this many blocks (small profiling case)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling slice of workload 2, 3 or 4: this many decoder layers, a small "
                         "vocabulary (and 8 experts for the MoE); same geometry and per-layer shapes")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--overlap", action="store_true",
                    help="measure the reduction overlapped with a simulated backward pass instead")
    ap.add_argument("--gemm", type=int, default=4096)
    ap.add_argument("--max-ctas", type=int, default=0, help="reduction grid cap in --overlap (0: all SMs)")
    ap.add_argument("--impl", default="grs", choices=["grs", "reference"])
    ap.add_argument("--soak", type=float, default=1.5, help="untimed seconds before timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", default="plain", choices=VARIANTS,
                    help="fp32-grads: fp32 rank gradients; unused: some tensors without a gradient "
                         "(masked norm and update); frozen: some tensors frozen at plan time")
    ap.add_argument("--checkpoint", action="store_true",
                    help="measure checkpoint restore with reshard (layout kernels + files) instead")
    ap.add_argument("--small", action="store_true",
                    help="the whole update in one launch (grs_update_small; plans of at most 128 tiles)")
    ap.add_argument("--graph", action="store_true",
                    help="replay the whole update as one captured CUDA graph (launch-bound workloads)")
    ap.add_argument("--micro", type=int, default=0,
                    help="override the workload's number of microbatches (distinct seeded gradients each)")
    ap.add_argument("--window", type=int, default=0,
                    help="trailing accumulation window: reduce only the first M' microbatches, G = acc/M'")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if args.workload is None and (args.variant != "plain" or args.graph or args.small or args.micro
                                  or args.overlap or args.checkpoint):
        args.workload = 1  # the variant rows and separate measurements are taken on the 67M plan
    if "WORLD_SIZE" not in os.environ and args.gpus > 1 and args.impl != "reference":
        # One process per GPU: start the ranks (torchrun) and pass on their status.
        sys.exit(subprocess.call(rank_launch_cmd(args.gpus, sys.argv[1:], _free_port())))
    rank = int(os.environ.get("RANK", "0"))
    world_size = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.impl == "reference" else 1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world_size)), flush=True)
        return
    if args.overlap:
        print(json.dumps(run_overlap(args)), flush=True)
        return
    if args.checkpoint:
        print(json.dumps(run_checkpoint(args)), flush=True)
        return
    if world_size > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_gpu(args, rank, world_size, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world_size > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
