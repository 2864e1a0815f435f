#!/usr/bin/env python3
"""Benchmark: ms per optimizer update (owner-routed reduce + clip + AdamW).

One step = one whole update over one batch of synthetic gradients: every
microbatch's reduction of all buckets (grs_reduce_all, norm partials fused
on the last microbatch), the global-norm finish (grs_grad_norm_sq) and the
fused clip + AdamW + bf16 cast (grs_clip_adamw_step).  Inputs are resident
in HBM and larger than L2 (each rank's gradient buffer alone exceeds it).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1]
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


def mandatory_bytes(op, n_micro: int, world: int) -> dict:
    """Algorithmic bytes of one update, per kernel.
    Per unique padded element with reduction group R_e: reduce reads
    2*M*R_e, writes acc 4 (first microbatch) or reads+writes 8 (later ones);
    the update reads acc, master, m, v (16) and writes master, m, v (12) and
    the bf16 parameter (2)."""
    red = 0
    n_state = 0
    for b in range(op.n_buckets):
        tag = int(op.b_tag[b])
        re = world if tag in (0, 1) else (op.dp if tag == 2 else 1)
        elems = op.copies(b) * int(op.b_padded[b])
        n_state += elems
        red += elems * (2 * n_micro * re + 4 + 8 * (n_micro - 1))
    return {"reduce": red, "update": 30 * n_state, "total": red + 30 * n_state,
            "reduce_last_mb": sum(op.copies(b) * int(op.b_padded[b]) *
                                  (2 * (world if int(op.b_tag[b]) in (0, 1) else
                                        (op.dp if int(op.b_tag[b]) == 2 else 1)) +
                                   (4 if n_micro == 1 else 8))
                                  for b in range(op.n_buckets))}


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
class GpuUpdate:
    """All device buffers of one workload and the three calls of one update."""

    def __init__(self, w: workloads.Workload, device):
        import torch
        from gradient_reduction_sharded_gb300 import grs
        self.torch, self.grs, self.w, self.dev = torch, grs, w, device
        self.plan = grs.grs_plan_create(w.numels, w.owners, w.world, w.tp, w.dp_replicate,
                                        w.dp_shard, w.bucket_bytes)
        self.info = grs.grs_plan_query(self.plan)
        nrp, nsp = self.info["n_rank_pad"], self.info["n_state_pad"]
        self.grads = [[workloads.normal_bf16(nrp, w.grad_std, workloads.grad_seed(w.cid, j, k),
                                             device=device)
                       for k in range(w.world)] for j in range(w.n_micro)]
        self.ptrs = [[t.data_ptr() for t in mb] for mb in self.grads]
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
        self.op = None
        self.step_no = 0
        # kernels per step: one reduction per microbatch, the norm finish, the update
        self.launches_per_step = w.n_micro + 2

    def reduce(self):
        g, w = self.grs, self.w
        for j in range(w.n_micro):
            g.grs_reduce_all(self.plan, self.ptrs[j], self.acc.data_ptr(), int(j > 0),
                             int(j == w.n_micro - 1), self.ws.data_ptr(), self.stream)

    def norm_sq(self):
        self.grs.grs_grad_norm_sq(self.plan, self.acc.data_ptr(), self.w.n_micro,
                                  self.ws.data_ptr(), 1, self.norm.data_ptr(), self.stream)

    def adamw(self):
        a = self.w.adamw
        self.step_no += 1
        hp = self.grs.make_adamw(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm,
                                 self.step_no, self.w.n_micro)
        self.grs.grs_clip_adamw_step(self.plan, hp, self.norm.data_ptr(), self.acc.data_ptr(),
                                     self.master.data_ptr(), self.m.data_ptr(), self.v.data_ptr(),
                                     self.params.data_ptr(), self.stream)

    def step(self):
        self.reduce()
        self.norm_sq()
        self.adamw()

    def close(self):
        self.torch.cuda.synchronize(self.dev)
        self.grs.grs_plan_destroy(self.plan)


def run_gpu(args, rank, world_size, local_rank):
    import torch
    import oracle  # CPU baseline leg only
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    w = workloads.get(args.workload, args.blocks)
    op = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard,
                     w.bucket_bytes)
    mb = mandatory_bytes(op, w.n_micro, w.world)
    u = GpuUpdate(w, device)
    u.op = op
    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit()
                          else local_rank)
    clocks.start()
    dist = None
    if world_size > 1:
        import torch.distributed as dist
    # warm-up: the first step initialises the moments (timing sees a warm state)
    clocks.mark("load_start")
    for _ in range(args.warmup):
        u.step()
    torch.cuda.synchronize()
    # soak so that the clock samples see the steady state (untimed)
    t_soak = time.time()
    while time.time() - t_soak < args.soak:
        for _ in range(10):
            u.step()
        torch.cuda.synchronize()
    K = args.steps
    # Timed region: exactly K steps, back to back, no events in between.
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for _ in range(K):
        u.step()
    t_end.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    ms_step = max_over_ranks(total_ms / K, device)
    # Per-kernel durations for the roofline: a second region of K steps with
    # CUDA events between the kernels on the launching stream (the events
    # themselves cost a few microseconds per step, so they stay out of the
    # headline region).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        ev[i][0].record()
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

    # ---------------------------------------------------------------- gather
    gather = run_gather(u, args, torch)

    # ---------------------------------------------------------------- e2e
    e2e = None if args.no_e2e else run_e2e(u, args, torch)

    status = u.grs.grs_check_device_errors(u.plan, u.stream)
    u.close()

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    kern = {
        "reduce": {"ms": statistics.mean(red_ms), "ms_median": statistics.median(red_ms),
                   "bytes": mb["reduce"] / w.n_micro, "launches_per_step": w.n_micro},
        "update": {"ms": statistics.mean(upd_ms), "ms_median": statistics.median(upd_ms),
                   "bytes": mb["update"], "launches_per_step": 1},
        "norm": {"ms": statistics.mean(nrm_ms), "ms_median": statistics.median(nrm_ms), "bytes": None,
                 "launches_per_step": 1},
    }
    # reduce: average per launch over the microbatches of a step
    kern["reduce"]["ms_per_launch"] = kern["reduce"]["ms"] / w.n_micro
    kern["update"]["ms_per_launch"] = kern["update"]["ms"]
    dom = "reduce" if kern["reduce"]["ms"] >= kern["update"]["ms"] else "update"
    dk = kern[dom]
    achieved = dk["bytes"] / (dk["ms_per_launch"] * 1e-3) / 1e9
    traffic = load_traffic(dom, w)
    result = {
        "metric": METRIC, "value": job_value(ms_step, world_size), "unit": UNIT, "n_gpus": world_size,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(w.describe(), grad_dtype="bf16", l2="inputs larger than L2 (no flush)",
                       parallelism=f"replicas{world_size}" if world_size > 1 else "1 GPU, simulated ranks"),
        "achieved_gbs_total": mb["total"] / (ms_step * world_size * 1e-3) / 1e9 if world_size == 1
        else mb["total"] / (ms_step * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": dk["bytes"]},
        "kernels": {k: {kk: vv for kk, vv in v.items()} for k, v in kern.items()},
        "e2e": e2e,
        "gather": gather,
        "gpu_launches": u.launches_per_step * K,
        "kernel_timing": "second region of K steps with CUDA events between the kernels",
        "per_update_ms": {"median": statistics.median(upd_total), "min": upd_total[0],
                          "max": upd_total[-1],
                          "note": "second region, one update per event pair (events between kernels add a few us)"},
        "clocks": clk,
        "device_status": status,
    }
    if rank == 0 and world_size == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, op, mb, args)
    return result


def run_gather(u: GpuUpdate, args, torch):
    """grs_gather_params to per-tensor bf16 storage, timed on its own (not part
    of the update: parameters can also be used as views of the bucket-ordered
    buffer).  Algorithmic bytes: read + write 2 bytes per parameter."""
    w = u.w
    outs = [torch.empty(n, dtype=torch.int16, device=u.dev) for n in w.numels]
    ptrs = [t.data_ptr() for t in outs]
    for _ in range(3):
        u.grs.grs_gather_params(u.plan, u.params.data_ptr(), ptrs, u.stream)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        u.grs.grs_gather_params(u.plan, u.params.data_ptr(), ptrs, u.stream)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.steps
    nbytes = 4 * w.n_unique
    del outs
    return {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9}


def run_e2e(u: GpuUpdate, args, torch):
    """The same update through the public C ABI with host buffers:
    grs_step_from_host copies every step's gradients from pinned host memory
    (bucket by bucket, overlapped with the reductions), runs the update and
    reads the bf16 parameters and the squared norm back to the host."""
    w = u.w
    W, M = w.world, w.n_micro
    n = u.info["n_rank_pad"]
    host = [torch.empty(n, dtype=torch.int16).pin_memory() for _ in range(M * W)]
    for j in range(M):
        for k in range(W):
            host[j * W + k].copy_(u.grads[j][k].view(torch.int16))
    halves = 2 if M > 1 else 1
    stage = [torch.empty(n, dtype=torch.bfloat16, device=u.dev) for _ in range(halves * W)]
    stage_ptrs = [t.data_ptr() for t in stage] + [stage[0].data_ptr()] * ((2 - halves) * W)
    out_params = torch.empty(u.params.numel(), dtype=torch.int16).pin_memory()
    out_norm = torch.empty(1, dtype=torch.float64).pin_memory()
    h2d = 0
    op = u.op
    for b in range(op.n_buckets):
        nread = 1 if int(op.b_tag[b]) == 3 else W
        h2d += M * nread * int(op.b_padded[b]) * 2
    d2h = out_params.numel() * 2 + 8
    steps = max(3, min(args.steps, 10))
    a = w.adamw

    def one():
        u.step_no += 1
        hp = u.grs.make_adamw(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, u.step_no, M)
        u.grs.grs_step_from_host(u.plan, hp, [t.data_ptr() for t in host], stage_ptrs,
                                 u.acc.data_ptr(), u.master.data_ptr(), u.m.data_ptr(), u.v.data_ptr(),
                                 u.params.data_ptr(), u.ws.data_ptr(), u.norm.data_ptr(),
                                 out_params.data_ptr(), out_norm.data_ptr(), u.stream)

    one()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        one()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    del stage
    return {"value": ms, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_gbs": h2d / (ms * 1e-3) / 1e9, "steps": steps,
            "path": "grs_step_from_host: pinned host gradients, per-bucket H2D overlapped with the "
                    "reductions, bf16 parameters and norm read back"}


KERNEL_SOURCES = ("kernels_reduce.cu", "kernels_update.cu", "device.cuh", "internal.h", "launch.cuh")


def csrc_hash() -> str:
    """Hash of the sources that define the reduce and update kernels, to tell
    whether stored DRAM counters still apply."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gradient_reduction_sharded_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, w):
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
    ent = t.get(f"{kernel}:{w.name}")
    return None if ent is None else ent.get("bytes_per_launch")


# --------------------------------------------------------------------------- CPU arm
def _host_inputs(w, op, device=None):
    """The workload's gradients as host uint16 arrays, generated exactly as the
    GPU arm generates them (same seeds), one buffer per (microbatch, rank)."""
    import torch
    dev = device or ("cuda" if torch.cuda.is_available() else "cpu")
    out = []
    for j in range(w.n_micro):
        row = []
        for k in range(w.world):
            t = workloads.normal_bf16(op.n_rank_pad, w.grad_std, workloads.grad_seed(w.cid, j, k),
                                      device=dev)
            row.append(workloads.bf16_bits(t.cpu()))
            del t
        out.append(row)
    return out


def _oracle_sample(w, op, host, buckets, threads=1):
    """One oracle update restricted to `buckets` (reduce -> norm -> AdamW);
    with threads > 1 the buckets run in parallel (the oracle's C code drops
    the GIL) and the norm is still summed in bucket order."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    a_ = w.adamw
    hp = (a_.lr, a_.beta1, a_.beta2, a_.eps, a_.weight_decay)

    def red(b):
        ro, P = int(op.b_rank_off[b]), int(op.b_padded[b])
        g = np.stack([np.stack([h[ro:ro + P] for h in mb]) for mb in host])
        a = oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard, P,
                                 int(op.b_used[b]), g)
        return a, oracle.norm_sq(a, w.n_micro)

    def upd(args):
        b, a, c = args
        P = int(op.b_padded[b])
        z = np.zeros(P, np.float32)
        for t in range(op.copies(b)):
            oracle.adamw(a[t], int(op.b_used[b]), w.n_micro, c, hp, 1, z, z, z)

    with ThreadPoolExecutor(max(1, threads)) as ex:
        parts = list(ex.map(red, buckets))
        s = 0.0
        for _, ns in parts:
            s += ns
        c = oracle.clip_coef(s, w.adamw.max_norm)
        list(ex.map(upd, [(b, a, c) for b, (a, _) in zip(buckets, parts)]))
    return s


def _sample_buckets(op, frac_target=0.35):
    """Buckets of every tag, smallest-first per tag, until ~frac_target of the
    state elements are covered (a bounded sample of the same workload)."""
    total = op.n_state_pad
    chosen, acc = [], 0
    by_tag = {}
    for b in range(op.n_buckets):
        by_tag.setdefault(int(op.b_tag[b]), []).append(b)
    for tag, bs in sorted(by_tag.items()):
        chosen.append(bs[0])
        acc += op.copies(bs[0]) * int(op.b_padded[bs[0]])
    for b in range(op.n_buckets):
        if acc >= frac_target * total:
            break
        if b not in chosen:
            chosen.append(b)
            acc += op.copies(b) * int(op.b_padded[b])
    return sorted(chosen)


def _sample_bytes(op, buckets, n_micro, world):
    tot = 0
    for b in buckets:
        tag = int(op.b_tag[b])
        re = world if tag in (0, 1) else (op.dp if tag == 2 else 1)
        elems = op.copies(b) * int(op.b_padded[b])
        tot += elems * (2 * n_micro * re + 4 + 8 * (n_micro - 1) + 30)
    return tot


def cpu_baseline(w, op, mb, args, host=None, target_s=10.0):
    """The oracle as it stands, on this host: whole updates of the workload
    (every bucket: reduce -> norm -> AdamW), repeated until about target_s of
    CPU work, one thread; then the same with one thread per core (buckets in
    parallel)."""
    host = host if host is not None else _host_inputs(w, op)
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
            "all_cores": {"value": dtn * 1e3, "cores": nthr,
                          "note": f"one whole update, {min(nthr, op.n_buckets)} buckets in parallel"}}


def run_reference(args, rank, world_size):
    """The oracle as the reference arm, on host cores, rank 0 only."""
    import oracle
    w = workloads.get(args.workload, args.blocks)
    op = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard,
                     w.bucket_bytes)
    mb = mandatory_bytes(op, w.n_micro, w.world)
    host = _host_inputs(w, op)
    buckets = _sample_buckets(op, frac_target=0.0)  # one bucket per tag: a bounded step
    sb = _sample_bytes(op, buckets, w.n_micro, w.world)
    for _ in range(args.warmup):
        _oracle_sample(w, op, host, buckets)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_sample(w, op, host, buckets)
    dt = (time.perf_counter() - t0) / args.steps
    ms = dt * 1e3 * mb["total"] / sb
    sample = (f"each step: oracle update of buckets {buckets} of {op.n_buckets} "
              f"({sb / 1e9:.2f} of {mb['total'] / 1e9:.2f} GB), one thread, scaled by bytes")
    return {"metric": METRIC, "value": ms, "unit": UNIT, "n_gpus": world_size, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": dict(w.describe(), l2="host memory"),
            "cpu_baseline": {"value": ms, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": ms, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


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
    w = workloads.get(args.workload, args.blocks)
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=1, choices=workloads.ALL_IDS)
    ap.add_argument("--blocks", type=int, default=0,
                    help="shrink workload 1 to this many blocks (small profiling case)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--overlap", action="store_true",
                    help="measure the reduction overlapped with a simulated backward pass instead")
    ap.add_argument("--gemm", type=int, default=4096)
    ap.add_argument("--max-ctas", type=int, default=0, help="reduction grid cap in --overlap (0: all SMs)")
    ap.add_argument("--impl", default="grs", choices=["grs", "reference"])
    ap.add_argument("--soak", type=float, default=1.5, help="untimed seconds before timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world_size = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world_size)), flush=True)
        return
    if args.overlap:
        print(json.dumps(run_overlap(args)), flush=True)
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
