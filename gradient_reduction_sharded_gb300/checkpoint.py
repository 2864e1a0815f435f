"""Checkpoints of the sharded optimizer state, restorable under another plan.

What the pages fix ("Distributed Transformer Training" integration note,
"Optimizer and checkpoint semantics"; "refactor(distributed): establish
shared native TP replica ownership", "Preserved prototype and evidence";
"Cosmos 3 ... distributed parallelism", section 2):

* a checkpoint stores the optimizer shards together with the optimizer step
  and the parallel geometry;
* it is loadable only once its ``_SUCCESS`` manifest has been committed;
* asynchronous saves report write failures from ``wait()``;
* the dp_replicate replicas of a shard read the same shard file, so a
  checkpoint holds one file per (dp_shard index, tp index);
* restoring into another ownership layout is exact and the next update
  matches the uninterrupted one.

Layout.  Shard file (s, t) holds, for every bucket, the slice
[s * shard_len, (s+1) * shard_len) of bucket row t (LOCAL_SHARD buckets) or
row 0 (every other bucket, stored once, in the t = 0 file: tensor-parallel
ranks hold identical copies of it), for each state array (master, exp_avg,
exp_avg_sq, ...).  ``manifest.json`` records the writer's plan, the file
list with SHA-256 digests, the step counts and caller metadata;
``_SUCCESS`` is written last, after every file is flushed to disk.

Restore.  The writer's state is reassembled from its shard files, moved
into the canonical logical order with the writer's plan
(grs_state_to_logical) and into the reader's bucket layout with the
reader's plan (grs_state_from_logical), both CUDA kernels.  The logical
order does not depend on tp, dp_replicate, dp_shard, owner tags or bucket
size.  This module does host file I/O only; all layout arithmetic on the
device goes through the C ABI.
"""
from __future__ import annotations

import hashlib
import json
import os
import shutil
import tempfile
from concurrent.futures import Future, ThreadPoolExecutor
from dataclasses import asdict, dataclass, field
from typing import Dict, List, Optional

import numpy as np

MANIFEST = "manifest.json"
SUCCESS = "_SUCCESS"
FORMAT = "grs-sharded-state/1"
LOCAL_SHARD = 2


class CheckpointError(RuntimeError):
    pass


@dataclass
class PlanSpec:
    """Everything needed to rebuild a plan (its logical parameter list and
    geometry)."""
    numels: List[int]
    owners: List[int]
    tensor_flags: Optional[List[int]]
    world: int
    tp: int
    dp_replicate: int
    dp_shard: int
    bucket_bytes: int
    plan_flags: int = 0

    def create(self, host_only: bool = False) -> int:
        from . import grs
        flags = self.plan_flags | (grs.GRS_PLAN_HOST_ONLY if host_only else 0)
        return grs.grs_plan_create_ex(self.numels, self.owners, self.tensor_flags, self.world, self.tp,
                                      self.dp_replicate, self.dp_shard, self.bucket_bytes, flags)


def _buckets(plan: int):
    from . import grs
    info = grs.grs_plan_query(plan)
    return info, [grs.grs_bucket_info(plan, b) for b in range(info["n_buckets"])]


def shard_slices(plan: int) -> Dict[str, list]:
    """{file name: [(state offset, length), ...]} of every shard file."""
    info, buckets = _buckets(plan)
    out = {}
    for t in range(info["tp"]):
        for s in range(info["dp_shard"]):
            sl = []
            for d in buckets:
                ls = d["tag"] == LOCAL_SHARD
                if not ls and t != 0:
                    continue
                row = t if ls else 0
                L = d["shard_len"]
                if L:
                    sl.append((d["state_offset"] + row * d["padded"] + s * L, L))
            out[f"shard_s{s}_t{t}.bin"] = sl
    return out


def _io_threads() -> int:
    return max(1, min(8, os.cpu_count() or 1))


def write_shards(directory: str, plan: int, spec: PlanSpec, arrays: Dict[str, np.ndarray],
                 steps: dict, metadata: Optional[dict] = None) -> None:
    """Write host fp32 state arrays (bucket layout of `plan`) as shard files,
    the manifest, and finally _SUCCESS.  The directory is built under a
    temporary name and renamed into place, so a reader never sees a partial
    checkpoint with _SUCCESS."""
    info, _ = _buckets(plan)
    names = sorted(arrays)
    for nm in names:
        a = arrays[nm]
        if a.dtype != np.float32 or a.size < info["n_state_pad"]:
            raise CheckpointError(f"array {nm}: need float32 with {info['n_state_pad']} elements")
    parent = os.path.dirname(os.path.abspath(directory)) or "."
    os.makedirs(parent, exist_ok=True)
    if os.path.exists(os.path.join(directory, SUCCESS)):
        raise CheckpointError(f"{directory} already holds a committed checkpoint")
    tmp = tempfile.mkdtemp(prefix=".grs-ckpt-", dir=parent)

    def write_one(item):
        # one shard file, its digest taken from the bytes as they are written
        fname, sl = item
        h = hashlib.sha256()
        with open(os.path.join(tmp, fname), "wb") as f:
            for nm in names:
                a = arrays[nm].reshape(-1)
                for off, n in sl:
                    buf = memoryview(np.ascontiguousarray(a[off:off + n])).cast("B")
                    h.update(buf)
                    f.write(buf)
            f.flush()
            os.fsync(f.fileno())
        return fname, {"slices": sl, "sha256": h.hexdigest(), "bytes": int(sum(n for _, n in sl) * 4 * len(names))}

    try:
        # shard files in parallel (hashing and file writes release the GIL)
        with ThreadPoolExecutor(max_workers=_io_threads()) as ex:
            files = dict(ex.map(write_one, shard_slices(plan).items()))
        manifest = {"format": FORMAT, "plan": asdict(spec), "arrays": names, "files": files,
                    "n_state_pad": info["n_state_pad"], "steps": steps, "metadata": metadata or {}}
        with open(os.path.join(tmp, MANIFEST), "w") as f:
            json.dump(manifest, f)
            f.flush()
            os.fsync(f.fileno())
        if os.path.isdir(directory):
            shutil.rmtree(directory)
        os.replace(tmp, directory)
        with open(os.path.join(directory, SUCCESS), "w") as f:
            f.write("ok\n")
            f.flush()
            os.fsync(f.fileno())
    except BaseException:
        shutil.rmtree(tmp, ignore_errors=True)
        raise


def read_shards(directory: str):
    """(manifest, {name: host fp32 array in the writer's bucket layout}).
    Refuses a checkpoint without _SUCCESS or with a file whose digest does
    not match the manifest."""
    if not os.path.exists(os.path.join(directory, SUCCESS)):
        raise CheckpointError(f"{directory}: no {SUCCESS}: the checkpoint was never committed")
    with open(os.path.join(directory, MANIFEST)) as f:
        man = json.load(f)
    if man.get("format") != FORMAT:
        raise CheckpointError(f"{directory}: unknown format {man.get('format')!r}")
    names = man["arrays"]
    arrays = {nm: np.zeros(man["n_state_pad"], np.float32) for nm in names}

    def read_one(item):
        # one shard file: read once, digest checked on those bytes, scattered
        # into the writer's layout (files cover disjoint slices)
        fname, ent = item
        path = os.path.join(directory, fname)
        data = np.fromfile(path, dtype=np.uint8)
        if hashlib.sha256(memoryview(data)).hexdigest() != ent["sha256"]:
            raise CheckpointError(f"{path}: digest mismatch")
        if data.size % 4:
            raise CheckpointError(f"{path}: size does not match the manifest")
        vals = data.view(np.float32)
        pos = 0
        for nm in names:
            for off, n in ent["slices"]:
                if pos + n > vals.size:
                    raise CheckpointError(f"{path}: size does not match the manifest")
                arrays[nm][off:off + n] = vals[pos:pos + n]
                pos += n
        if pos != vals.size:
            raise CheckpointError(f"{path}: size does not match the manifest")

    with ThreadPoolExecutor(max_workers=_io_threads()) as ex:
        list(ex.map(read_one, man["files"].items()))
    return man, arrays


# ---------------------------------------------------------------------------- device side
def save(directory: str, plan: int, spec: PlanSpec, state: Dict[str, "object"], steps: dict,
         metadata: Optional[dict] = None) -> None:
    """Save device fp32 state arrays (torch tensors in `plan`'s layout)."""
    host = {nm: t.detach().float().cpu().numpy() for nm, t in state.items()}
    write_shards(directory, plan, spec, host, steps, metadata)


class _Saving:
    def __init__(self, fut: Future):
        self._fut = fut

    def wait(self):
        """Block until the files are written; re-raise any write failure."""
        return self._fut.result()

    def done(self) -> bool:
        return self._fut.done()


_pool = ThreadPoolExecutor(max_workers=1, thread_name_prefix="grs-ckpt")


def save_async(directory: str, plan: int, spec: PlanSpec, state: Dict[str, "object"], steps: dict,
               metadata: Optional[dict] = None) -> _Saving:
    """Copy the device state to host memory now (so training may go on and
    overwrite it), write the files in the background; ``wait()`` returns when
    the checkpoint is committed and raises if writing failed."""
    host = {nm: t.detach().float().cpu().numpy() for nm, t in state.items()}
    return _Saving(_pool.submit(write_shards, directory, plan, spec, host, steps, metadata))


def load(directory: str, plan: int, out: Dict[str, "object"], stream: Optional[int] = None) -> dict:
    """Restore into device fp32 arrays `out` (torch tensors in `plan`'s bucket
    layout, possibly another geometry or ownership than the writer's).
    Returns the manifest (steps, metadata, writer plan)."""
    import torch

    from . import grs
    man, arrays = read_shards(directory)
    spec = PlanSpec(**man["plan"])
    writer = spec.create()
    try:
        winfo = grs.grs_plan_query(writer)
        rinfo = grs.grs_plan_query(plan)
        if winfo["n_unique"] != rinfo["n_unique"]:
            raise CheckpointError("the checkpoint's logical parameters do not match the plan's "
                                  f"({winfo['n_unique']} vs {rinfo['n_unique']} elements)")
        dev = next(iter(out.values())).device
        s = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream
        logical = torch.empty(max(1, winfo["n_unique"]), dtype=torch.float32, device=dev)
        for nm, dst in out.items():
            if nm not in arrays:
                raise CheckpointError(f"array {nm} not in the checkpoint")
            src = torch.from_numpy(arrays[nm]).to(dev)
            grs.grs_state_to_logical(writer, src.data_ptr(), logical.data_ptr(), s)
            grs.grs_state_from_logical(plan, logical.data_ptr(), dst.data_ptr(), s)
        torch.cuda.synchronize(dev)
    finally:
        grs.grs_plan_destroy(writer)
    return man
