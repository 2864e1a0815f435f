"""Shared helpers of the GPU parity tests: seeded inputs on the device, the
CUDA path through the C ABI, the oracle on the same bytes, comparisons.

Inputs come from `workloads` (seeded torch generators); expected values come
only from `oracle` applied to those inputs copied to the host.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

import oracle
import workloads

NAN_BF16 = 0x7FC0
RTOL, ATOL = 1e-5, 1e-7


def grs():
    from gradient_reduction_sharded_gb300 import grs as g
    return g


@dataclass
class Case:
    """A plan plus the device buffers of one update."""
    numels: List[int]
    owners: List[int]
    world: int
    tp: int
    dp_replicate: int
    dp_shard: int
    bucket_bytes: int
    n_micro: int
    grad_std: float
    seed_base: int
    hp: tuple = (1e-3, 0.9, 0.999, 1e-8, 0.01)
    max_norm: float = 1.0
    master_std: float = 0.02
    fp32_grads: bool = False
    tensor_flags: Optional[List[int]] = None


def case_from_workload(cid: int) -> Case:
    w = workloads.get(cid)
    a = w.adamw
    return Case(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes,
                w.n_micro, w.grad_std, cid, (a.lr, a.beta1, a.beta2, a.eps, a.weight_decay),
                a.max_norm, w.master_std)


class Run:
    """Device-side state of one case: plan, rank buffers per microbatch,
    accumulator, optimizer state, workspace."""

    def __init__(self, c: Case, device="cuda", poison_padding=True, step_seed=0):
        g = grs()
        self.c = c
        self.dev = torch.device(device)
        self.op = oracle.plan(c.numels, c.owners, c.world, c.tp, c.dp_replicate, c.dp_shard,
                              c.bucket_bytes, c.tensor_flags)
        flags = g.GRS_PLAN_FP32_GRADS if c.fp32_grads else 0
        self.plan = g.grs_plan_create_ex(c.numels, c.owners, c.tensor_flags, c.world, c.tp,
                                         c.dp_replicate, c.dp_shard, c.bucket_bytes, flags)
        self.info = g.grs_plan_query(self.plan)
        nrp, nsp = self.info["n_rank_pad"], self.info["n_state_pad"]
        self.nrp, self.nsp = nrp, nsp
        self.poison = poison_padding
        gdt = torch.float32 if c.fp32_grads else torch.bfloat16
        self.grads = [[torch.empty(max(nrp, 8), dtype=gdt, device=self.dev)
                       for _ in range(c.world)] for _ in range(c.n_micro)]
        self.fill_grads(step_seed)
        self.acc = torch.empty(max(nsp, 8), dtype=torch.float32, device=self.dev)
        self.master = workloads.normal_f32(max(nsp, 8), c.master_std,
                                           workloads.master_seed(c.seed_base), device=self.dev)
        self.m = torch.zeros(max(nsp, 8), dtype=torch.float32, device=self.dev)
        self.v = torch.zeros(max(nsp, 8), dtype=torch.float32, device=self.dev)
        self.params = self.master.to(torch.bfloat16).view(torch.int16).clone()
        self.ws = torch.zeros(max(self.info["workspace_bytes"], 16) // 4 + 4, dtype=torch.float32,
                              device=self.dev)
        self.norm = torch.zeros(1, dtype=torch.float64, device=self.dev)
        self.step = 0

    def fill_grads(self, step_seed=0):
        c = self.c
        for j in range(c.n_micro):
            for k in range(c.world):
                seed = workloads.grad_seed(c.seed_base, j + 1000 * step_seed, k)
                if c.fp32_grads:
                    workloads.normal_f32(self.nrp, c.grad_std, seed, device=self.dev,
                                         out=self.grads[j][k][:self.nrp])
                else:
                    workloads.normal_bf16(self.nrp, c.grad_std, seed, device=self.dev,
                                          out=self.grads[j][k][:self.nrp])
                if self.poison:
                    for b in range(self.op.n_buckets):
                        ro = int(self.op.b_rank_off[b])
                        lo, hi = ro + int(self.op.b_used[b]), ro + int(self.op.b_padded[b])
                        if c.fp32_grads:
                            self.grads[j][k][lo:hi] = float("nan")
                        else:
                            self.grads[j][k].view(torch.int16)[lo:hi] = NAN_BF16

    def stream(self) -> int:
        return torch.cuda.current_stream(self.dev).cuda_stream

    def ptrs(self, j):
        return [t.data_ptr() for t in self.grads[j]]

    def reduce(self, per_bucket=False, emit=True, n_micro=None):
        g = grs()
        c = self.c
        s = self.stream()
        M = c.n_micro if n_micro is None else n_micro
        for j in range(M):
            last = emit and j == M - 1
            if per_bucket:
                for b in range(self.info["n_buckets"]):
                    d = g.grs_bucket_info(self.plan, b)
                    rp = [p + 2 * d["rank_offset"] for p in self.ptrs(j)]
                    g.grs_reduce_bucket(self.plan, b, rp, self.acc.data_ptr() + 4 * d["state_offset"],
                                        int(j > 0), int(last), self.ws.data_ptr(), s)
            else:
                g.grs_reduce_all(self.plan, self.ptrs(j), self.acc.data_ptr(), int(j > 0), int(last),
                                 self.ws.data_ptr(), s)

    def norm_sq(self, partials_ready=True):
        g = grs()
        g.grs_grad_norm_sq(self.plan, self.acc.data_ptr(), self.c.n_micro, self.ws.data_ptr(),
                           int(partials_ready), self.norm.data_ptr(), self.stream())

    def adamw(self, max_norm=None):
        g = grs()
        c = self.c
        self.step += 1
        mn = c.max_norm if max_norm is None else max_norm
        hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], mn, self.step, c.n_micro)
        g.grs_clip_adamw_step(self.plan, hp, self.norm.data_ptr(), self.acc.data_ptr(),
                              self.master.data_ptr(), self.m.data_ptr(), self.v.data_ptr(),
                              self.params.data_ptr(), self.stream())

    def update(self, per_bucket=False, partials_ready=True, max_norm=None):
        self.reduce(per_bucket=per_bucket, emit=partials_ready)
        self.norm_sq(partials_ready=partials_ready)
        self.adamw(max_norm=max_norm)

    def masked_reduce(self, used_dev, emit=True, n_micro=None):
        """grs_reduce_all_masked over the microbatches; with emit, the last
        one writes the masked norm partials into the workspace."""
        g = grs()
        M = self.c.n_micro if n_micro is None else n_micro
        for j in range(M):
            g.grs_reduce_all_masked(self.plan, self.ptrs(j), self.acc.data_ptr(), int(j > 0),
                                    int(emit and j == M - 1), used_dev.data_ptr(), self.ws.data_ptr(),
                                    self.stream())

    def masked_norm_separate(self, used_dev, n_micro=None):
        """S from the separate masked norm pass over acc, into a new buffer
        (the workspace's partials are overwritten)."""
        out = torch.zeros(1, dtype=torch.float64, device=self.dev)
        M = self.c.n_micro if n_micro is None else n_micro
        grs().grs_grad_norm_sq_masked(self.plan, self.acc.data_ptr(), M, used_dev.data_ptr(),
                                      self.ws.data_ptr(), out.data_ptr(), self.stream())
        return out

    def masked_update(self, used_dev, steps_dev, n_micro=None, max_norm=None, step_hint=1,
                      partials_ready=False):
        """Norm over used tensors and the per-tensor-step AdamW (the reduce
        must have run).  partials_ready: the masked reduction emitted the
        norm partials, so only the finish runs (grs_grad_norm_sq); otherwise
        the separate masked norm pass.  step_hint goes in hp->step: tensors
        whose new step equals it use host-computed factors, the others
        device-computed ones."""
        g = grs()
        c = self.c
        M = c.n_micro if n_micro is None else n_micro
        mn = c.max_norm if max_norm is None else max_norm
        s = self.stream()
        if partials_ready:
            g.grs_grad_norm_sq(self.plan, self.acc.data_ptr(), M, self.ws.data_ptr(), 1,
                               self.norm.data_ptr(), s)
        else:
            g.grs_grad_norm_sq_masked(self.plan, self.acc.data_ptr(), M, used_dev.data_ptr(),
                                      self.ws.data_ptr(), self.norm.data_ptr(), s)
        hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], mn, step_hint, M)
        g.grs_clip_adamw_step_masked(self.plan, hp, self.norm.data_ptr(), self.acc.data_ptr(),
                                     self.master.data_ptr(), self.m.data_ptr(), self.v.data_ptr(),
                                     self.params.data_ptr(), used_dev.data_ptr(), steps_dev.data_ptr(),
                                     self.ws.data_ptr(), s)

    def check_flags(self) -> int:
        return grs().grs_check_device_errors(self.plan, self.stream())

    def close(self):
        if self.plan:
            torch.cuda.synchronize(self.dev)
            g = grs()
            if g.grs_build_features() & g.GRS_FEATURE_CHECKED:
                # checked build: no kernel may have left a buffer
                st = g.grs_check_device_errors(self.plan, self.stream())
                assert st != g.GRS_ERR_BOUNDS, g.grs_last_error()
            g.grs_plan_destroy(self.plan)
            self.plan = None

    # ---------------------------------------------------------------- oracle side
    def bucket_inputs(self, b) -> np.ndarray:
        """[M][R][P] of bucket b copied to the host: uint16 bf16 bits, or
        float32 for fp32-gradient plans."""
        ro = int(self.op.b_rank_off[b])
        P = int(self.op.b_padded[b])
        arr = torch.stack([torch.stack([t[ro:ro + P] for t in mb]) for mb in self.grads])
        if self.c.fp32_grads:
            return arr.cpu().numpy()
        return arr.view(torch.int16).cpu().numpy().view(np.uint16)

    def state_host(self):
        n = self.nsp
        return (self.master[:n].cpu().numpy().copy(), self.m[:n].cpu().numpy().copy(),
                self.v[:n].cpu().numpy().copy())


def oracle_update(run: Run, master0, m0, v0, step: int, max_norm=None, threads=1):
    c = run.c
    mn = c.max_norm if max_norm is None else max_norm
    return oracle.full_update(run.op, run.bucket_inputs, c.n_micro, c.hp, mn, step, master0, m0, v0,
                              threads=threads, bounds=True)


def assert_close(got, want, what, rtol=RTOL, atol=ATOL):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    both_nan = np.isnan(got) & np.isnan(want)
    err = np.abs(got - want)
    bad = ~both_nan & ~(err <= atol + rtol * np.abs(want))
    if bad.any():
        i = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside rel {rtol}/abs {atol}; "
                             f"first {i.tolist()} got {got[i].tolist()} want {want[i].tolist()}")


# At most this fraction of the elements of one comparison (and at least
# BRACKET_MIN_COUNT) may need the bracket below to pass: the bracket exists
# for the rare ill-conditioned AdamW points, and a systematic error that it
# would hide must still fail.
BRACKET_MAX_FRACTION = 1e-4
BRACKET_MIN_COUNT = 2


def bracket_cap(n: int) -> int:
    return max(BRACKET_MIN_COUNT, int(np.ceil(BRACKET_MAX_FRACTION * n)))


def assert_close_bracketed(got, want, lo, hi, what, rtol=RTOL, atol=ATOL):
    """rel/abs tolerance around the oracle's value, widened to the bracket
    [min(lo, hi), max(lo, hi)] of the oracle's update at acc -/+ the fp32
    accumulation error bound.  Away from ill-conditioned points the bracket
    is far inside the tolerance; where AdamW's g / (|g| + eps) magnifies the
    rounding an fp32 accumulator must make, it is what the arithmetic allows.
    Only bracket_cap(n) elements may fall outside the plain tolerance;
    returns how many did."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    a = np.asarray(lo, np.float64)
    b = np.asarray(hi, np.float64)
    lo = np.minimum(np.minimum(a, b), want)
    hi = np.maximum(np.maximum(a, b), want)
    both_nan = np.isnan(got) & np.isnan(want)
    tol = atol + rtol * np.abs(want)
    bad = ~both_nan & ~((got >= lo - tol) & (got <= hi + tol))
    if bad.any():
        i = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside the bracketed tolerance; first "
                             f"{i.tolist()} got {got[i].tolist()} want {want[i].tolist()} "
                             f"bracket {lo[i].tolist()}..{hi[i].tolist()}")
    n_out = int((~both_nan & ((got < want - tol) | (got > want + tol))).sum())
    assert n_out <= bracket_cap(got.size), (
        f"{what}: {n_out} of {got.size} elements needed the accumulation bracket "
        f"(at most {bracket_cap(got.size)} may)")
    return n_out


def assert_within_accumulation_bound(got_acc, want_acc, delta, what):
    """The fp32 accumulator against the oracle's exact (fp64) one: the
    difference may not exceed the accumulation error bound delta that widens
    the master and moment checks, element by element (NaN where both are
    NaN)."""
    got = np.asarray(got_acc, np.float64)
    want = np.asarray(want_acc, np.float64)
    d = np.asarray(delta, np.float64)
    both_nan = np.isnan(got) & np.isnan(want)
    bad = ~both_nan & ~(np.abs(got - want) <= d)
    if bad.any():
        i = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} accumulator values beyond the fp32 accumulation "
                             f"bound; first {i.tolist()} got {got[i].tolist()} want {want[i].tolist()} "
                             f"bound {d[i].tolist()}")


def bf16_ordered(bits):
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_value(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_bf16_cast(got_bits, got_master, want_bits, want_master, what, rtol=RTOL, atol=ATOL,
                     lo_master=None, hi_master=None):
    """bf16 parameters.  (1) The kernel's bf16 is the round-to-nearest-even of
    its own fp32 master, bit for bit (torch's CPU cast decides, in fp32).
    (2) Against the oracle: within 1 bf16 ulp, widened by the fp32 master
    tolerance where the masters themselves may differ by that much (values
    near zero, where a bf16 ulp is far below abs 1e-7), and by the master's
    bracket when one is given (the oracle's update at acc -/+ the fp32
    accumulation bound: at ill-conditioned AdamW points the masters may
    differ by more than a bf16 ulp, and the casts with them)."""
    g = np.asarray(got_bits).view(np.uint16)
    w = np.asarray(want_bits, np.uint16)
    rne = torch.from_numpy(np.asarray(got_master, np.float32)).to(torch.bfloat16)
    rne = rne.view(torch.int16).numpy().view(np.uint16)
    gn = np.isnan(bf16_value(g))
    bad = (g != rne) & ~gn
    assert not bad.any(), f"{what}: bf16 is not the RNE of the fp32 master at {np.flatnonzero(bad)[:5]}"
    wn = np.isnan(bf16_value(w))
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    gv, wv = bf16_value(g), bf16_value(w)
    ulp = np.abs(bf16_value(w ^ 1) - wv)  # spacing at the oracle's value
    lim = ulp + atol + rtol * np.abs(np.asarray(want_master, np.float64))
    d = np.abs(gv - wv)
    if lo_master is not None and hi_master is not None:
        # distance from the cast to the cast interval of the bracket
        wm = np.asarray(want_master, np.float64)
        a = np.minimum(np.minimum(np.asarray(lo_master, np.float64), np.asarray(hi_master, np.float64)), wm)
        b = np.maximum(np.maximum(np.asarray(lo_master, np.float64), np.asarray(hi_master, np.float64)), wm)
        d = np.minimum(d, np.maximum(0.0, np.maximum(a - gv, gv - b)))
    d[gn] = 0
    if (d > lim).any():
        i = np.flatnonzero(d > lim)[:5]
        raise AssertionError(f"{what}: {int((d > lim).sum())} bf16 values beyond tolerance at "
                             f"{i.tolist()}: got {g[i].tolist()} want {w[i].tolist()}")


def padding_mask(op) -> np.ndarray:
    """True at state elements that are padding."""
    mask = np.zeros(op.n_state_pad, bool)
    for b in range(op.n_buckets):
        P = int(op.b_padded[b])
        for t in range(op.copies(b)):
            o = int(op.b_state_off[b]) + t * P
            mask[o + int(op.b_used[b]):o + P] = True
    return mask
