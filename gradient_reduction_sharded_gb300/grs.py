"""Thin ctypes binding of libgrs (include/grs.h), same names as the C ABI.

Argument marshalling only: device pointers are passed as Python ints
(e.g. ``tensor.data_ptr()``) and streams as ``torch.cuda.Stream.cuda_stream``
ints.  Every computation happens in libgrs's CUDA kernels; if the library
is missing this module raises at import time — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
# GRS_LIBRARY may name another build of the same library (e.g. a variant
# compiled with different tile constants); default: the in-tree build.
LIB_PATH = os.environ.get("GRS_LIBRARY") or os.path.join(_HERE, "libgrs.so")

GRS_REPLICA_AVG, GRS_PARTIAL_SUM, GRS_LOCAL_SHARD, GRS_ALREADY_REDUCED = 0, 1, 2, 3
GRS_OK = 0
GRS_ERR_INVALID_ARG = 1
GRS_ERR_UNSUPPORTED_COMPOSITION = 2
GRS_ERR_SHAPE = 3
GRS_ERR_ALIGNMENT = 4
GRS_ERR_CUDA = 5
GRS_ERR_TIMEOUT = 6
GRS_ERR_NONFINITE = 7
GRS_ERR_NO_DEVICE = 8
GRS_ERR_BOUNDS = 9
GRS_FEATURE_CHECKED = 1
GRS_PLAN_HOST_ONLY = 1
GRS_PLAN_FP32_GRADS = 2
GRS_TENSOR_FROZEN = 1
GRS_MAX_WORLD = 128
GRS_NOALLOC_SCRATCH_BYTES = 4 << 20
GRS_SMALL_MAX_TILES = 128
GRS_SMALL_MAX_BUFFERS = 256

STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED_COMPOSITION", 3: "SHAPE",
                4: "ALIGNMENT", 5: "CUDA", 6: "TIMEOUT", 7: "NONFINITE", 8: "NO_DEVICE",
                9: "BOUNDS"}


class GrsError(RuntimeError):
    def __init__(self, status: int, func: str, msg: str):
        super().__init__(f"{func}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class grs_plan_info(ctypes.Structure):
    _fields_ = [("n_tensors", ctypes.c_int32), ("n_buckets", ctypes.c_int32),
                ("world", ctypes.c_int32), ("tp", ctypes.c_int32),
                ("dp_replicate", ctypes.c_int32), ("dp_shard", ctypes.c_int32),
                ("dp", ctypes.c_int32), ("device", ctypes.c_int32),
                ("n_unique", ctypes.c_int64), ("n_rank_pad", ctypes.c_int64),
                ("n_state_pad", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("n_reduce_tiles", ctypes.c_int64), ("grad_bytes", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class grs_bucket_desc(ctypes.Structure):
    _fields_ = [("tag", ctypes.c_int32), ("copies", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("n_tensors", ctypes.c_int32),
                ("used", ctypes.c_int64), ("padded", ctypes.c_int64),
                ("shard_len", ctypes.c_int64), ("rank_offset", ctypes.c_int64),
                ("state_offset", ctypes.c_int64), ("n_segments", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class grs_segment_desc(ctypes.Structure):
    _fields_ = [("tensor", ctypes.c_int32), ("tp_index", ctypes.c_int32),
                ("bucket_offset", ctypes.c_int64), ("tensor_offset", ctypes.c_int64),
                ("numel", ctypes.c_int64), ("state_offset", ctypes.c_int64)]


class grs_tensor_desc(ctypes.Structure):
    _fields_ = [("bucket", ctypes.c_int32), ("owner", ctypes.c_int32),
                ("numel", ctypes.c_int64), ("per_rank", ctypes.c_int64),
                ("bucket_offset", ctypes.c_int64), ("flags", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


class grs_adamw(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("max_norm", ctypes.c_float), ("step", ctypes.c_int32),
                ("n_micro", ctypes.c_int32)]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                      "(there is no CPU fallback)")
_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_P = ctypes.POINTER
_sig = {
    "grs_plan_create": ([_P(ctypes.c_int64), _P(ctypes.c_int32), ctypes.c_int32, ctypes.c_int32,
                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                         ctypes.c_uint32, _P(_vp)], ctypes.c_int),
    "grs_plan_create_ex": ([_P(ctypes.c_int64), _P(ctypes.c_int32), _P(ctypes.c_uint32), ctypes.c_int32,
                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                            ctypes.c_int64, ctypes.c_uint32, _P(_vp)], ctypes.c_int),
    "grs_plan_destroy": ([_vp], None),
    "grs_plan_shard_view": ([_vp, ctypes.c_int32, ctypes.c_int32, _P(_vp)], ctypes.c_int),
    "grs_plan_query": ([_vp, _P(grs_plan_info)], ctypes.c_int),
    "grs_bucket_info": ([_vp, ctypes.c_int32, _P(grs_bucket_desc)], ctypes.c_int),
    "grs_tensor_info": ([_vp, ctypes.c_int32, _P(grs_tensor_desc)], ctypes.c_int),
    "grs_segment_info": ([_vp, ctypes.c_int32, ctypes.c_int32, _P(grs_segment_desc)], ctypes.c_int),
    "grs_reduce_bucket": ([_vp, ctypes.c_int32, _P(_vp), _vp, ctypes.c_int32, ctypes.c_int32, _vp,
                           _vp], ctypes.c_int),
    "grs_reduce_all": ([_vp, _P(_vp), _vp, ctypes.c_int32, ctypes.c_int32, _vp, _vp], ctypes.c_int),
    "grs_reduce_bucket_ex": ([_vp, ctypes.c_int32, _P(_vp), _vp, ctypes.c_int32, ctypes.c_int32, _vp,
                              ctypes.c_int32, _vp, _vp], ctypes.c_int),
    "grs_reduce_all_masked": ([_vp, _P(_vp), _vp, ctypes.c_int32, ctypes.c_int32, _vp, _vp, _vp], ctypes.c_int),
    "grs_accumulate": ([_vp, ctypes.c_int32, _vp, _vp, _vp], ctypes.c_int),
    "grs_grad_norm_sq": ([_vp, _vp, ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp], ctypes.c_int),
    "grs_clip_adamw_step": ([_vp, _P(grs_adamw), _vp, _vp, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "grs_gather_params": ([_vp, _vp, _P(_vp), _vp], ctypes.c_int),
    "grs_clip_adamw_step_to_tensors": ([_vp, _P(grs_adamw), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
                                       ctypes.c_int),
    "grs_grad_norm_sq_masked": ([_vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp], ctypes.c_int),
    "grs_clip_adamw_step_masked": ([_vp, _P(grs_adamw), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _vp], ctypes.c_int),
    "grs_check_device_errors": ([_vp, _vp], ctypes.c_int),
    "grs_selftest_bounded_wait": ([_vp, ctypes.c_int64, _vp], ctypes.c_int),
    "grs_check_already_reduced": ([_vp, _P(_vp), _vp], ctypes.c_int),
    "grs_state_to_logical": ([_vp, _vp, _vp, _vp], ctypes.c_int),
    "grs_state_from_logical": ([_vp, _vp, _vp, _vp], ctypes.c_int),
    "grs_grad_norm_sq_noalloc": ([_vp, _vp, ctypes.c_int32, _vp, _vp], ctypes.c_int),
    "grs_step_from_host": ([_vp, _P(grs_adamw), _P(_vp), _P(_vp), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                            _vp, _vp, _vp], ctypes.c_int),
    "grs_update_small": ([_vp, _P(grs_adamw), _P(_vp), _vp, _vp, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "grs_last_error": ([], ctypes.c_char_p),
    "grs_build_features": ([], ctypes.c_uint32),
}
for _name, (_args, _res) in _sig.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_sig)


def grs_last_error() -> str:
    return (_lib.grs_last_error() or b"").decode()


def grs_build_features() -> int:
    return int(_lib.grs_build_features())


def _check(status: int, func: str):
    if status != GRS_OK:
        raise GrsError(status, func, grs_last_error())


def pointer_array(seq: Sequence[Optional[int]]):
    """A reusable C array of device pointers: every call below that takes a
    pointer list also takes one of these as is (no conversion per call)."""
    return _ptrs(seq)


def _ptrs(seq: Sequence[Optional[int]]):
    if isinstance(seq, ctypes.Array):
        return seq
    arr = (_vp * max(1, len(seq)))()
    for i, p in enumerate(seq):
        arr[i] = None if p is None else int(p)
    return arr


def grs_plan_create(numels: Sequence[int], owners: Sequence[int], world: int, tp: int,
                    dp_replicate: int, dp_shard: int, bucket_bytes: int, flags: int = 0) -> int:
    n = len(numels)
    ne = (ctypes.c_int64 * max(1, n))(*numels)
    ow = (ctypes.c_int32 * max(1, n))(*owners)
    out = _vp()
    _check(_lib.grs_plan_create(ne, ow, n, world, tp, dp_replicate, dp_shard, bucket_bytes, flags,
                                ctypes.byref(out)), "grs_plan_create")
    return out.value


def grs_plan_create_ex(numels: Sequence[int], owners: Sequence[int], tensor_flags: Optional[Sequence[int]],
                       world: int, tp: int, dp_replicate: int, dp_shard: int, bucket_bytes: int,
                       flags: int = 0) -> int:
    n = len(numels)
    ne = (ctypes.c_int64 * max(1, n))(*numels)
    ow = (ctypes.c_int32 * max(1, n))(*owners)
    tf = None if tensor_flags is None else (ctypes.c_uint32 * max(1, n))(*tensor_flags)
    out = _vp()
    _check(_lib.grs_plan_create_ex(ne, ow, tf, n, world, tp, dp_replicate, dp_shard, bucket_bytes,
                                   flags, ctypes.byref(out)), "grs_plan_create_ex")
    return out.value


def grs_plan_shard_view(plan: int, shard: int, tp_index: int) -> int:
    out = _vp()
    _check(_lib.grs_plan_shard_view(plan, shard, tp_index, ctypes.byref(out)), "grs_plan_shard_view")
    return out.value


def grs_plan_destroy(plan: int) -> None:
    _lib.grs_plan_destroy(plan)


def _as_dict(s) -> Dict[str, int]:
    return {k: getattr(s, k) for k, _ in s._fields_}


def grs_plan_query(plan: int) -> Dict[str, int]:
    o = grs_plan_info()
    _check(_lib.grs_plan_query(plan, ctypes.byref(o)), "grs_plan_query")
    return _as_dict(o)


def grs_bucket_info(plan: int, bucket: int) -> Dict[str, int]:
    o = grs_bucket_desc()
    _check(_lib.grs_bucket_info(plan, bucket, ctypes.byref(o)), "grs_bucket_info")
    return _as_dict(o)


def grs_tensor_info(plan: int, tensor: int) -> Dict[str, int]:
    o = grs_tensor_desc()
    _check(_lib.grs_tensor_info(plan, tensor, ctypes.byref(o)), "grs_tensor_info")
    return _as_dict(o)


def grs_segment_info(plan: int, bucket: int, segment: int) -> Dict[str, int]:
    o = grs_segment_desc()
    _check(_lib.grs_segment_info(plan, bucket, segment, ctypes.byref(o)), "grs_segment_info")
    return _as_dict(o)


def grs_reduce_bucket(plan: int, bucket: int, rank_grads: Sequence[int], acc: int, accumulate: int,
                      emit_norm_partials: int, workspace: Optional[int], stream: int) -> None:
    _check(_lib.grs_reduce_bucket(plan, bucket, _ptrs(rank_grads), acc, accumulate,
                                  emit_norm_partials, workspace, stream), "grs_reduce_bucket")


def grs_reduce_bucket_ex(plan: int, bucket: int, rank_grads: Sequence[int], acc: int, accumulate: int,
                         emit_norm_partials: int, workspace: Optional[int], max_ctas: int,
                         wait_event: Optional[int], stream: int) -> None:
    """wait_event: a cudaEvent_t handle (torch.cuda.Event.cuda_event) or None."""
    _check(_lib.grs_reduce_bucket_ex(plan, bucket, _ptrs(rank_grads), acc, accumulate,
                                     emit_norm_partials, workspace, max_ctas, wait_event, stream),
           "grs_reduce_bucket_ex")


def grs_reduce_all(plan: int, rank_grads: Sequence[int], acc: int, accumulate: int,
                   emit_norm_partials: int, workspace: Optional[int], stream: int) -> None:
    _check(_lib.grs_reduce_all(plan, _ptrs(rank_grads), acc, accumulate, emit_norm_partials,
                               workspace, stream), "grs_reduce_all")


def grs_reduce_all_masked(plan: int, rank_grads: Sequence[int], acc: int, accumulate: int,
                          emit_norm_partials: int, d_tensor_used: int, workspace: Optional[int],
                          stream: int) -> None:
    _check(_lib.grs_reduce_all_masked(plan, _ptrs(rank_grads), acc, accumulate, emit_norm_partials,
                                      d_tensor_used, workspace, stream), "grs_reduce_all_masked")


def grs_accumulate(plan: int, bucket: int, acc: int, mb: int, stream: int) -> None:
    _check(_lib.grs_accumulate(plan, bucket, acc, mb, stream), "grs_accumulate")


def grs_grad_norm_sq(plan: int, acc: Optional[int], n_micro: int, workspace: int,
                     partials_ready: int, d_norm_sq: int, stream: int) -> None:
    _check(_lib.grs_grad_norm_sq(plan, acc, n_micro, workspace, partials_ready, d_norm_sq, stream),
           "grs_grad_norm_sq")


def make_adamw(lr, beta1, beta2, eps, weight_decay, max_norm, step, n_micro) -> grs_adamw:
    return grs_adamw(lr, beta1, beta2, eps, weight_decay, max_norm, step, n_micro)


def grs_clip_adamw_step(plan: int, hp: grs_adamw, d_norm_sq: Optional[int], acc: int, master: int,
                        m: int, v: int, params_bf16: int, stream: int) -> None:
    _check(_lib.grs_clip_adamw_step(plan, ctypes.byref(hp), d_norm_sq, acc, master, m, v,
                                    params_bf16, stream), "grs_clip_adamw_step")


def grs_clip_adamw_step_to_tensors(plan: int, hp: grs_adamw, d_norm_sq: Optional[int], acc: int,
                                   master: int, m: int, v: int, params_bf16: Optional[int],
                                   d_tensor_ptrs: int, stream: int) -> None:
    """d_tensor_ptrs: device address of an int64 array of per-tensor device
    pointers (0 = skip), e.g. ``torch.tensor(ptrs, dtype=torch.int64,
    device=...).data_ptr()``."""
    _check(_lib.grs_clip_adamw_step_to_tensors(plan, ctypes.byref(hp), d_norm_sq, acc, master, m, v,
                                               params_bf16, d_tensor_ptrs, stream),
           "grs_clip_adamw_step_to_tensors")


def grs_gather_params(plan: int, params_bf16: int, tensor_ptrs: Sequence[Optional[int]],
                      stream: int) -> None:
    _check(_lib.grs_gather_params(plan, params_bf16, _ptrs(tensor_ptrs), stream),
           "grs_gather_params")


def grs_step_from_host(plan: int, hp: grs_adamw, host_grads: Sequence[int], dev_stage: Sequence[int],
                       acc: int, master: int, m: int, v: int, params_bf16: int, workspace: int,
                       d_norm_sq: int, host_params: Optional[int], host_norm_sq: Optional[int],
                       stream: int) -> None:
    _check(_lib.grs_step_from_host(plan, ctypes.byref(hp), _ptrs(host_grads), _ptrs(dev_stage), acc,
                                   master, m, v, params_bf16, workspace, d_norm_sq, host_params,
                                   host_norm_sq, stream), "grs_step_from_host")


def grs_grad_norm_sq_noalloc(plan: int, acc: int, n_micro: int, d_norm_sq: int, stream: int) -> None:
    """Global squared norm with the library's static scratch (no workspace,
    no allocation); for callers that cannot allocate device memory."""
    _check(_lib.grs_grad_norm_sq_noalloc(plan, acc, n_micro, d_norm_sq, stream),
           "grs_grad_norm_sq_noalloc")


def grs_grad_norm_sq_masked(plan: int, acc: int, n_micro: int, d_tensor_used: int, workspace: int,
                            d_norm_sq: int, stream: int) -> None:
    _check(_lib.grs_grad_norm_sq_masked(plan, acc, n_micro, d_tensor_used, workspace, d_norm_sq, stream),
           "grs_grad_norm_sq_masked")


def grs_clip_adamw_step_masked(plan: int, hp: grs_adamw, d_norm_sq: Optional[int], acc: int, master: int,
                               m: int, v: int, params_bf16: int, d_tensor_used: int, d_tensor_steps: int,
                               workspace: int, stream: int) -> None:
    _check(_lib.grs_clip_adamw_step_masked(plan, ctypes.byref(hp), d_norm_sq, acc, master, m, v,
                                           params_bf16, d_tensor_used, d_tensor_steps, workspace, stream),
           "grs_clip_adamw_step_masked")


def grs_update_small(plan: int, hp: grs_adamw, rank_grads: Sequence[int], acc: int, master: int, m: int,
                     v: int, params_bf16: int, d_norm_sq: int, stream: int) -> None:
    """The whole update of a small plan in one launch; rank_grads holds
    n_micro * world buffers, microbatch-major."""
    _check(_lib.grs_update_small(plan, ctypes.byref(hp), _ptrs(rank_grads), acc, master, m, v, params_bf16,
                                 d_norm_sq, stream), "grs_update_small")


def grs_state_to_logical(plan: int, state: int, logical: int, stream: int) -> None:
    _check(_lib.grs_state_to_logical(plan, state, logical, stream), "grs_state_to_logical")


def grs_state_from_logical(plan: int, logical: int, state: int, stream: int) -> None:
    _check(_lib.grs_state_from_logical(plan, logical, state, stream), "grs_state_from_logical")


def grs_check_already_reduced(plan: int, rank_grads: Sequence[int], stream: int) -> None:
    _check(_lib.grs_check_already_reduced(plan, _ptrs(rank_grads), stream), "grs_check_already_reduced")


def grs_selftest_bounded_wait(plan: int, limit_ns: int, stream: int) -> None:
    _check(_lib.grs_selftest_bounded_wait(plan, limit_ns, stream), "grs_selftest_bounded_wait")


def grs_check_device_errors(plan: int, stream: int) -> int:
    """Returns the status (raises only for CUDA errors)."""
    st = _lib.grs_check_device_errors(plan, stream)
    if st == GRS_ERR_CUDA:
        _check(st, "grs_check_device_errors")
    return st
