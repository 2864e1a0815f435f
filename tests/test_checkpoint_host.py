"""Checkpoint file layer on the host (no GPU): shard files per (dp_shard,
tp) index shared by replicas, manifest with digests, _SUCCESS last,
refusals, asynchronous save reporting failures from wait()."""
import os

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def grs():
    from gradient_reduction_sharded_gb300 import _build
    _build.build()
    from gradient_reduction_sharded_gb300 import grs as g
    return g


@pytest.fixture(scope="module")
def ck():
    from gradient_reduction_sharded_gb300 import checkpoint
    return checkpoint


def spec_of(ck, **kw):
    base = dict(numels=[21, 5, 18, 3, 1000, 64], owners=[0, 1, 2, 3, 0, 2], tensor_flags=None, world=8,
                tp=2, dp_replicate=2, dp_shard=2, bucket_bytes=1024, plan_flags=0)
    base.update(kw)
    return ck.PlanSpec(**base)


def test_round_trip_and_layout(tmp_path, grs, ck):
    spec = spec_of(ck)
    plan = spec.create(host_only=True)
    try:
        n = grs.grs_plan_query(plan)["n_state_pad"]
        rng = np.random.default_rng(3)
        arrays = {nm: rng.normal(0, 1, n).astype(np.float32) for nm in ("master", "exp_avg", "exp_avg_sq")}
        op = oracle.plan(spec.numels, spec.owners, spec.world, spec.tp, spec.dp_replicate, spec.dp_shard,
                         spec.bucket_bytes)
        # padding is not state: zero it so the round trip is exact
        pad = np.ones(n, bool)
        for b in range(op.n_buckets):
            for t in range(op.copies(b)):
                o = int(op.b_state_off[b]) + t * int(op.b_padded[b])
                pad[o:o + int(op.b_used[b])] = False
        for a in arrays.values():
            a[pad] = 0
        d = str(tmp_path / "ck1")
        ck.write_shards(d, plan, spec, arrays, {"step": 7}, {"note": "x"})
        files = sorted(f for f in os.listdir(d) if f.startswith("shard_"))
        # one file per (dp_shard, tp) index; the dp_replicate replicas share them
        assert files == sorted(f"shard_s{s}_t{t}.bin" for s in range(2) for t in range(2))
        man, back = ck.read_shards(d)
        assert man["steps"] == {"step": 7} and man["metadata"] == {"note": "x"}
        for nm in arrays:
            assert np.array_equal(back[nm], arrays[nm])
        # every state element is in exactly one file
        cover = np.zeros(n, int)
        for ent in man["files"].values():
            for off, ln in ent["slices"]:
                cover[off:off + ln] += 1
        assert np.all(cover == 1)
        with pytest.raises(ck.CheckpointError):
            ck.write_shards(d, plan, spec, arrays, {"step": 8})  # already committed
    finally:
        grs.grs_plan_destroy(plan)


def test_refuses_uncommitted_or_corrupt(tmp_path, grs, ck):
    spec = spec_of(ck)
    plan = spec.create(host_only=True)
    try:
        n = grs.grs_plan_query(plan)["n_state_pad"]
        arrays = {"master": np.ones(n, np.float32)}
        d = str(tmp_path / "ck2")
        ck.write_shards(d, plan, spec, arrays, {"step": 1})
        os.remove(os.path.join(d, ck.SUCCESS))
        with pytest.raises(ck.CheckpointError, match="never committed"):
            ck.read_shards(d)
        d3 = str(tmp_path / "ck3")
        ck.write_shards(d3, plan, spec, arrays, {"step": 1})
        with open(os.path.join(d3, "shard_s1_t0.bin"), "r+b") as f:
            f.seek(4)
            f.write(b"\x00\x00\x80\x7f")
        with pytest.raises(ck.CheckpointError, match="digest"):
            ck.read_shards(d3)
    finally:
        grs.grs_plan_destroy(plan)


def test_async_save_reports_failure_from_wait(tmp_path, grs, ck):
    spec = spec_of(ck)
    plan = spec.create(host_only=True)
    try:
        n = grs.grs_plan_query(plan)["n_state_pad"]
        blocker = tmp_path / "file"
        blocker.write_text("not a directory")
        fut = ck._pool.submit(ck.write_shards, str(blocker / "ck"), plan, spec,
                              {"master": np.ones(n, np.float32)}, {"step": 1})
        with pytest.raises(Exception):
            ck._Saving(fut).wait()
        ok = ck._Saving(ck._pool.submit(ck.write_shards, str(tmp_path / "ck4"), plan, spec,
                                        {"master": np.ones(n, np.float32)}, {"step": 1}))
        ok.wait()
        assert os.path.exists(os.path.join(str(tmp_path / "ck4"), ck.SUCCESS))
    finally:
        grs.grs_plan_destroy(plan)


def test_many_shard_files_in_parallel(tmp_path, grs, ck):
    """24 shard files (tp 2 x dp_shard 12), more than the I/O threads: every
    file written and read back exactly; a truncated file is refused."""
    spec = spec_of(ck, numels=[4001, 77, 960, 9, 123456, 24], world=24, tp=2, dp_replicate=1, dp_shard=12,
                   bucket_bytes=4096)
    plan = spec.create(host_only=True)
    try:
        n = grs.grs_plan_query(plan)["n_state_pad"]
        op = oracle.plan(spec.numels, spec.owners, spec.world, spec.tp, spec.dp_replicate, spec.dp_shard,
                         spec.bucket_bytes)
        keep = np.zeros(n, bool)
        for b in range(op.n_buckets):
            for t in range(op.copies(b)):
                o = int(op.b_state_off[b]) + t * int(op.b_padded[b])
                keep[o:o + int(op.b_used[b])] = True
        rng = np.random.default_rng(11)
        arrays = {nm: np.where(keep, rng.normal(0, 1, n), 0).astype(np.float32)
                  for nm in ("master", "exp_avg", "exp_avg_sq")}
        d = str(tmp_path / "many")
        ck.write_shards(d, plan, spec, arrays, {"step": 3})
        files = sorted(f for f in os.listdir(d) if f.startswith("shard_"))
        assert len(files) == 24
        _, back = ck.read_shards(d)
        for nm in arrays:
            assert np.array_equal(back[nm], arrays[nm])
        victim = os.path.join(d, "shard_s7_t1.bin")
        with open(victim, "r+b") as f:
            f.truncate(os.path.getsize(victim) - 4)
        with pytest.raises(ck.CheckpointError):
            ck.read_shards(d)
    finally:
        grs.grs_plan_destroy(plan)
