"""ctypes binding for the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
benchmark's CPU-baseline leg load this module; the product path never does.
The binding marshals numpy arrays; every step of the arithmetic is in
oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_COMPOSITION, ERR_SHAPE = 0, 1, 2, 3
REPLICA_AVG, PARTIAL_SUM, LOCAL_SHARD, ALREADY_REDUCED = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain C11, -O2, no
    fast-math, no FMA contraction)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                          os.path.getmtime(os.path.join(_HERE, "oracle.h"))))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")


def load_library(path: str):
    """ctypes handle of an oracle shared library with every signature set."""
    L = ctypes.CDLL(path)
    L.oracle_resolve_dims.argtypes = [ctypes.c_int32] * 4 + [_i32p]
    L.oracle_resolve_dims.restype = ctypes.c_int
    L.oracle_plan.argtypes = [_i64p, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                              _i32p, _i32p, _i64p, _i32p, _i64p, _i64p, _i64p, _i64p]
    L.oracle_plan.restype = ctypes.c_int
    L.oracle_plan_ex.argtypes = [_i64p, _i32p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                 ctypes.c_int32, _i32p, _i32p, _i64p, _i32p, _i64p, _i64p,
                                 _i64p, _i64p]
    L.oracle_plan_ex.restype = ctypes.c_int
    L.oracle_rank.argtypes = [ctypes.c_int32] * 5
    L.oracle_rank.restype = ctypes.c_int32
    L.oracle_reduce_bucket.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_int64, ctypes.c_int64,
                                                              ctypes.c_int32, _u16p, _f64p]
    L.oracle_reduce_bucket.restype = ctypes.c_int
    L.oracle_reduce_bucket_f32.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_int64, ctypes.c_int64,
                                                                  ctypes.c_int32, _f32p, _f64p]
    L.oracle_reduce_bucket_f32.restype = ctypes.c_int
    L.oracle_norm_sq.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int32]
    L.oracle_norm_sq.restype = ctypes.c_double
    L.oracle_clip_coef.argtypes = [ctypes.c_double, ctypes.c_double]
    L.oracle_clip_coef.restype = ctypes.c_double
    L.oracle_adamw.argtypes = [ctypes.c_int64, ctypes.c_int64, _f64p, ctypes.c_int32,
                               ctypes.c_double, _f64p, ctypes.c_int32,
                               _f32p, _f32p, _f32p, _f32p, _f32p, _f32p, _u16p]
    L.oracle_adamw.restype = None
    L.oracle_bf16_rne.argtypes = [ctypes.c_float]
    L.oracle_bf16_rne.restype = ctypes.c_uint16
    L.oracle_gather_tensor.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       _u16p, _u16p]
    L.oracle_gather_tensor.restype = None
    for nm in ("oracle_gather_tensor_f32", "oracle_scatter_tensor_f32"):
        f = getattr(L, nm)
        f.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                      ctypes.c_int64, ctypes.c_int64, _f32p, _f32p]
        f.restype = None
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB_PATH)
    return _lib


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


@dataclass
class OraclePlan:
    numel: np.ndarray
    owner: np.ndarray
    world: int
    tp: int
    dp_replicate: int
    dp_shard: int
    dp: int
    bucket_bytes: int
    t_bucket: np.ndarray
    t_offset: np.ndarray
    b_tag: np.ndarray
    b_padded: np.ndarray
    b_used: np.ndarray
    b_rank_off: np.ndarray
    b_state_off: np.ndarray

    @property
    def n_buckets(self) -> int:
        return int(self.b_tag.shape[0])

    def copies(self, b: int) -> int:
        return self.tp if int(self.b_tag[b]) == LOCAL_SHARD else 1

    @property
    def n_rank_pad(self) -> int:
        return int(self.b_padded.sum())

    @property
    def n_state_pad(self) -> int:
        return int(sum(self.copies(b) * int(self.b_padded[b]) for b in range(self.n_buckets)))

    def shard_len(self, b: int) -> int:
        return int(self.b_padded[b]) // self.dp_shard

    def per_rank(self, i: int) -> int:
        if int(self.t_bucket[i]) < 0:
            return 0
        n = int(self.numel[i])
        return n // self.tp if int(self.owner[i]) == LOCAL_SHARD else n

    def tensor_rows(self, i: int):
        """State ranges [lo, hi) of tensor i, one per bucket row."""
        b = int(self.t_bucket[i])
        if b < 0:
            return []
        P, o, n = int(self.b_padded[b]), int(self.t_offset[i]), self.per_rank(i)
        return [(int(self.b_state_off[b]) + t * P + o, int(self.b_state_off[b]) + t * P + o + n)
                for t in range(self.copies(b))]


def plan(numels: Sequence[int], owners: Sequence[int], world: int, tp: int, dp_replicate: int,
         dp_shard: int, bucket_bytes: int, tensor_flags: Optional[Sequence[int]] = None) -> OraclePlan:
    L = lib()
    n = len(numels)
    numel = np.ascontiguousarray(numels, dtype=np.int64)
    owner = np.ascontiguousarray(owners, dtype=np.int32)
    maxb = max(1, n)
    dims = np.zeros(4, np.int32)
    tb = np.zeros(max(1, n), np.int32)
    to = np.zeros(max(1, n), np.int64)
    btag = np.zeros(maxb, np.int32)
    bpad = np.zeros(maxb, np.int64)
    bused = np.zeros(maxb, np.int64)
    broff = np.zeros(maxb, np.int64)
    bsoff = np.zeros(maxb, np.int64)
    if n == 0:
        numel = np.zeros(1, np.int64)
        owner = np.zeros(1, np.int32)
    fl = None
    if tensor_flags is not None:
        fl_arr = np.ascontiguousarray(list(tensor_flags) or [0], dtype=np.uint32)
        fl = fl_arr.ctypes.data_as(ctypes.c_void_p)
    st = L.oracle_plan_ex(numel, owner, fl, n, world, tp, dp_replicate, dp_shard, bucket_bytes, maxb,
                          dims, tb, to, btag, bpad, bused, broff, bsoff)
    if st != OK:
        raise OracleError(st, "oracle_plan")
    nb = int(dims[3])
    return OraclePlan(numel[:n].copy(), owner[:n].copy(), world, tp, dp_replicate, int(dims[0]),
                      int(dims[1]), bucket_bytes, tb[:n].copy(), to[:n].copy(), btag[:nb].copy(),
                      bpad[:nb].copy(), bused[:nb].copy(), broff[:nb].copy(), bsoff[:nb].copy())


def rank(r: int, s: int, t: int, dp_shard: int, tp: int) -> int:
    return int(lib().oracle_rank(r, s, t, dp_shard, tp))


def reduce_bucket(tag: int, tp: int, dp_replicate: int, dp_shard: int, P: int, used: int,
                  grads: np.ndarray) -> np.ndarray:
    """grads: [M][R][P] uint16 (bf16 bits) or float32 -> fp64 acc [copies][P]."""
    f32 = np.asarray(grads).dtype == np.float32
    grads = np.ascontiguousarray(grads, dtype=np.float32 if f32 else np.uint16)
    M = grads.shape[0]
    R = tp * dp_replicate * dp_shard
    assert grads.shape == (M, R, P), (grads.shape, (M, R, P))
    copies = tp if tag == LOCAL_SHARD else 1
    acc = np.zeros((copies, P), np.float64)
    g = grads.reshape(-1) if grads.size else np.zeros(1, grads.dtype)
    a = acc.reshape(-1) if acc.size else np.zeros(1)
    fn = lib().oracle_reduce_bucket_f32 if f32 else lib().oracle_reduce_bucket
    st = fn(tag, tp, dp_replicate, dp_shard, P, used, M, g, a)
    if st != OK:
        raise OracleError(st, "oracle_reduce_bucket")
    return acc


def norm_sq(acc: np.ndarray, M: int) -> float:
    a = np.ascontiguousarray(acc, dtype=np.float64).reshape(-1)
    if a.size == 0:
        return 0.0
    return float(lib().oracle_norm_sq(a, a.size, M))


def clip_coef(norm_sq_value: float, max_norm: float) -> float:
    return float(lib().oracle_clip_coef(norm_sq_value, max_norm))


def bf16_rne(x: float) -> int:
    return int(lib().oracle_bf16_rne(x))


def adamw(acc: np.ndarray, used: int, M: int, c: float, hp, step: int,
          master0: np.ndarray, m0: np.ndarray, v0: np.ndarray):
    """One AdamW step over one unit.  hp = (lr, beta1, beta2, eps, wd).
    Returns (master1, m1, v1, bf16 bits)."""
    acc = np.ascontiguousarray(acc, dtype=np.float64).reshape(-1)
    n = acc.size
    master0 = np.ascontiguousarray(master0, dtype=np.float32).reshape(-1)
    m0 = np.ascontiguousarray(m0, dtype=np.float32).reshape(-1)
    v0 = np.ascontiguousarray(v0, dtype=np.float32).reshape(-1)
    out = [np.zeros(max(1, n), np.float32) for _ in range(3)]
    bits = np.zeros(max(1, n), np.uint16)
    if n:
        lib().oracle_adamw(n, used, acc, M, c, np.asarray(hp, np.float64), step, master0, m0, v0,
                           out[0], out[1], out[2], bits)
    return out[0][:n], out[1][:n], out[2][:n], bits[:n]


def gather_tensor(p: OraclePlan, i: int, params_full: np.ndarray) -> np.ndarray:
    b = int(p.t_bucket[i])
    n = int(p.numel[i])
    dst = np.zeros(max(1, n), np.uint16)
    src = np.ascontiguousarray(params_full, dtype=np.uint16).reshape(-1)
    if n:
        lib().oracle_gather_tensor(n, int(p.owner[i]), p.tp, int(p.b_state_off[b]),
                                   int(p.b_padded[b]), int(p.t_offset[i]), src, dst)
    return dst[:n]


def to_logical(p: OraclePlan, state: np.ndarray) -> np.ndarray:
    """fp32 state in bucket layout -> canonical logical order (live tensors in
    model order, each over its full logical extent)."""
    state = np.ascontiguousarray(state, dtype=np.float32).reshape(-1)
    parts = []
    for i in range(len(p.numel)):
        b = int(p.t_bucket[i])
        if b < 0:
            continue
        n = int(p.numel[i])
        dst = np.zeros(max(1, n), np.float32)
        if n:
            lib().oracle_gather_tensor_f32(n, int(p.owner[i]), p.tp, int(p.b_state_off[b]),
                                           int(p.b_padded[b]), int(p.t_offset[i]), state, dst)
        parts.append(dst[:n])
    return np.concatenate(parts) if parts else np.zeros(0, np.float32)


def from_logical(p: OraclePlan, logical: np.ndarray) -> np.ndarray:
    """Canonical logical order -> fp32 state in bucket layout (padding 0)."""
    logical = np.ascontiguousarray(logical, dtype=np.float32).reshape(-1)
    state = np.zeros(max(1, p.n_state_pad), np.float32)
    pos = 0
    for i in range(len(p.numel)):
        b = int(p.t_bucket[i])
        if b < 0:
            continue
        n = int(p.numel[i])
        if n:
            src = np.ascontiguousarray(logical[pos:pos + n])
            lib().oracle_scatter_tensor_f32(n, int(p.owner[i]), p.tp, int(p.b_state_off[b]),
                                            int(p.b_padded[b]), int(p.t_offset[i]), src, state)
        pos += n
    return state[:p.n_state_pad]


# ---------------------------------------------------------------------------
# Whole-update helper built from the functions above, in the pages' order:
# reduce every bucket (all microbatches) -> global norm -> clip coefficient
# -> AdamW per unit.  `grads_of(b)` returns the bucket's [M][R][P] uint16
# inputs; state arrays are full [n_state_pad] fp32.
# ---------------------------------------------------------------------------
@dataclass
class UpdateResult:
    acc: np.ndarray       # fp64 [n_state_pad]
    norm_sq: float
    clip: float
    master: np.ndarray
    m: np.ndarray
    v: np.ndarray
    params_bf16: np.ndarray
    # Optional brackets of master, m, v: the update evaluated at acc - delta
    # and acc + delta, delta bounding an fp32 evaluation's accumulation error
    # (see accumulation_error_bound), and delta itself [n_state_pad].
    lo: Optional[tuple] = None
    hi: Optional[tuple] = None
    delta: Optional[np.ndarray] = None


U32 = 2.0 ** -24  # unit roundoff of fp32


def abs_inputs(g: np.ndarray) -> np.ndarray:
    """|g| elementwise: bf16 bits with the sign cleared, or np.abs of fp32."""
    g = np.asarray(g)
    return np.abs(g) if g.dtype == np.float32 else (g & np.uint16(0x7FFF))


def gamma(k: int) -> float:
    """Higham's gamma_k = k u / (1 - k u) for fp32 (u = 2^-24): the bound on
    the relative perturbation that k roundings can put on one term."""
    return k * U32 / (1.0 - k * U32)


def group_terms(p: OraclePlan, b: int) -> int:
    """Ranks summed into one output element of bucket b per microbatch: the
    whole world for REPLICA_AVG and PARTIAL_SUM, the DP group for
    LOCAL_SHARD, rank 0 alone for ALREADY_REDUCED."""
    tag = int(p.b_tag[b])
    return p.world if tag in (REPLICA_AVG, PARTIAL_SUM) else (p.dp if tag == LOCAL_SHARD else 1)


def accumulation_error_bound(acc_abs: np.ndarray, M: int, group: int) -> np.ndarray:
    """Forward error bound of an fp32 evaluation of one accumulator element:
    per microbatch, the `group` rank values summed by recursive fp32
    addition in any order (group - 1 roundings; a compensated sum stays
    inside the same bound), multiplied by the tag's scale held in fp32 (one
    rounding of the constant, one of the product) and added into the fp32
    accumulator (one rounding per later microbatch, two if the multiply and
    add are not fused).  Every term then carries at most group + M + 1
    roundings, so |fl(acc) - acc| <= gamma_{group+M+1} * sum |terms|, where
    acc_abs is the same reduction of the absolute inputs, i.e. sum |terms|
    (Higham, Accuracy and Stability of Numerical Algorithms, 2nd ed.,
    Lemma 3.1 and section 4.2 on recursive summation)."""
    return gamma(group + M + 1) * acc_abs


def full_update(p: OraclePlan, grads_of, M: int, hp, max_norm: float, step: int,
                master0: np.ndarray, m0: np.ndarray, v0: np.ndarray,
                threads: int = 1, bounds: bool = False) -> UpdateResult:
    nsp = p.n_state_pad
    acc = np.zeros(nsp, np.float64)
    delta = np.zeros(nsp, np.float64) if bounds else None

    def red(b):
        P = int(p.b_padded[b])
        g = grads_of(b)
        a = reduce_bucket(int(p.b_tag[b]), p.tp, p.dp_replicate, p.dp_shard, P, int(p.b_used[b]), g)
        off = int(p.b_state_off[b])
        acc[off:off + a.size] = a.reshape(-1)
        if bounds:
            ab = reduce_bucket(int(p.b_tag[b]), p.tp, p.dp_replicate, p.dp_shard, P, int(p.b_used[b]),
                               abs_inputs(g))
            delta[off:off + ab.size] = accumulation_error_bound(ab.reshape(-1), M, group_terms(p, b))

    if threads > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(red, range(p.n_buckets)))
    else:
        for b in range(p.n_buckets):
            red(b)
    s = norm_sq(acc, M)
    c = clip_coef(s, max_norm)

    def update(a):
        master = np.zeros(nsp, np.float32)
        mm = np.zeros(nsp, np.float32)
        vv = np.zeros(nsp, np.float32)
        bits = np.zeros(nsp, np.uint16)
        for b in range(p.n_buckets):
            P = int(p.b_padded[b])
            for t in range(p.copies(b)):
                o = int(p.b_state_off[b]) + t * P
                r = adamw(a[o:o + P], int(p.b_used[b]), M, c, hp, step,
                          master0[o:o + P], m0[o:o + P], v0[o:o + P])
                master[o:o + P], mm[o:o + P], vv[o:o + P], bits[o:o + P] = r
        return master, mm, vv, bits

    master, mm, vv, bits = update(acc)
    res = UpdateResult(acc, s, c, master, mm, vv, bits)
    if bounds:
        res.lo = update(acc - delta)[:3]
        res.hi = update(acc + delta)[:3]
        res.delta = delta
    return res


def full_update_masked(p: OraclePlan, grads_of, M: int, hp, max_norm: float, used, steps,
                       master0: np.ndarray, m0: np.ndarray, v0: np.ndarray, params0: np.ndarray,
                       threads: int = 1, bounds: bool = True):
    """One update where tensor i has a gradient iff used[i] (PyTorch's grad
    None otherwise): the norm sums used tensors only (clip_grad_norm_ skips
    the others), and AdamW advances only used tensors, each with its own
    step count (steps[i] before this update; torch.optim.AdamW keeps one per
    parameter).  Unused tensors keep master, moments and bf16 copy.
    Returns the result (with brackets when `bounds`) and the new step counts."""
    nsp = p.n_state_pad
    acc = np.zeros(nsp, np.float64)
    delta = np.zeros(nsp, np.float64)
    for b in range(p.n_buckets):
        P = int(p.b_padded[b])
        g = grads_of(b)
        a = reduce_bucket(int(p.b_tag[b]), p.tp, p.dp_replicate, p.dp_shard, P, int(p.b_used[b]), g)
        off = int(p.b_state_off[b])
        acc[off:off + a.size] = a.reshape(-1)
        if bounds:
            ab = reduce_bucket(int(p.b_tag[b]), p.tp, p.dp_replicate, p.dp_shard, P, int(p.b_used[b]),
                               abs_inputs(g))
            delta[off:off + ab.size] = accumulation_error_bound(ab.reshape(-1), M, group_terms(p, b))
    s = 0.0
    for i in range(len(p.numel)):
        if used[i]:
            for lo, hi in p.tensor_rows(i):
                s += norm_sq(acc[lo:hi], M)
    c = clip_coef(s, max_norm)
    new_steps = list(steps)
    for i in range(len(p.numel)):
        if p.tensor_rows(i) and used[i]:
            new_steps[i] = steps[i] + 1

    def update(a):
        master = np.zeros(nsp, np.float32)
        mm = np.zeros(nsp, np.float32)
        vv = np.zeros(nsp, np.float32)
        bits = np.zeros(nsp, np.uint16)
        for i in range(len(p.numel)):
            for lo, hi in p.tensor_rows(i):
                if used[i]:
                    r = adamw(a[lo:hi], hi - lo, M, c, hp, new_steps[i], master0[lo:hi], m0[lo:hi],
                              v0[lo:hi])
                    master[lo:hi], mm[lo:hi], vv[lo:hi], bits[lo:hi] = r
                else:
                    master[lo:hi], mm[lo:hi], vv[lo:hi] = master0[lo:hi], m0[lo:hi], v0[lo:hi]
                    bits[lo:hi] = params0[lo:hi]
        return master, mm, vv, bits

    master, mm, vv, bits = update(acc)
    res = UpdateResult(acc, s, c, master, mm, vv, bits)
    if bounds:
        res.lo = update(acc - delta)[:3]
        res.hi = update(acc + delta)[:3]
        res.delta = delta
    return res, new_steps
