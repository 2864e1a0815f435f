"""Host-side checks of libgrs (no GPU): exports, plan tables against the
oracle's independent plan (bit-exact), rejections, host-only behaviour."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def grs():
    from gradient_reduction_sharded_gb300 import _build
    _build.build()
    from gradient_reduction_sharded_gb300 import grs as g
    return g


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(grs_[a-z0-9_]+)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(grs):
    names = declared_functions()
    assert "grs_reduce_bucket" in names and "grs_clip_adamw_step" in names
    lib = ctypes.CDLL(grs.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding wraps every declared function
    assert set(names) <= set(grs.EXPORTED), set(names) - set(grs.EXPORTED)


def test_default_build_is_not_the_checked_one(grs):
    if os.environ.get("GRS_LIBRARY"):
        pytest.skip("another build of the library is loaded")
    assert grs.grs_build_features() & grs.GRS_FEATURE_CHECKED == 0


def _compare_plan(grs, h, op, numels, owners):
    info = grs.grs_plan_query(h)
    assert info["n_buckets"] == op.n_buckets
    assert info["dp_shard"] == op.dp_shard
    assert info["dp"] == op.dp
    assert info["n_rank_pad"] == op.n_rank_pad
    assert info["n_state_pad"] == op.n_state_pad
    assert info["n_unique"] == int(sum(n for i, n in enumerate(numels) if int(op.t_bucket[i]) >= 0))
    for b in range(op.n_buckets):
        d = grs.grs_bucket_info(h, b)
        assert d["tag"] == int(op.b_tag[b])
        assert d["used"] == int(op.b_used[b])
        assert d["padded"] == int(op.b_padded[b])
        assert d["rank_offset"] == int(op.b_rank_off[b])
        assert d["state_offset"] == int(op.b_state_off[b])
        assert d["shard_len"] == op.shard_len(b)
        assert d["copies"] == op.copies(b)
    for i in range(len(numels)):
        t = grs.grs_tensor_info(h, i)
        assert t["bucket"] == int(op.t_bucket[i])
        assert t["bucket_offset"] == int(op.t_offset[i])
        assert t["numel"] == numels[i]
        assert t["owner"] == owners[i]
    _compare_segments(grs, h, op, numels)


def _compare_segments(grs, h, op, numels):
    """Segments against the oracle's tensor placement: row by row, the
    bucket's tensors in model order, each at the oracle's offset and state
    range; together they tile [0, used) of every row and cover every live
    tensor's elements exactly once."""
    covered = {i: 0 for i in range(len(numels)) if int(op.t_bucket[i]) >= 0}
    for b in range(op.n_buckets):
        members = [i for i in range(len(numels)) if int(op.t_bucket[i]) == b]
        d = grs.grs_bucket_info(h, b)
        assert d["n_segments"] == op.copies(b) * len(members)
        for t in range(op.copies(b)):
            pos = 0
            for k, i in enumerate(members):
                s = grs.grs_segment_info(h, b, t * len(members) + k)
                assert s["tensor"] == i and s["tp_index"] == t
                assert s["bucket_offset"] == int(op.t_offset[i]) == pos
                assert s["numel"] == op.per_rank(i)
                assert s["tensor_offset"] == t * op.per_rank(i)
                assert s["state_offset"] == op.tensor_rows(i)[t][0]
                pos += s["numel"]
                covered[i] += s["numel"]
            assert pos == int(op.b_used[b])
        with pytest.raises(grs.GrsError):
            grs.grs_segment_info(h, b, d["n_segments"])
        with pytest.raises(grs.GrsError):
            grs.grs_segment_info(h, b, -1)
    assert all(covered[i] == numels[i] for i in covered)


@pytest.mark.parametrize("cid", workloads.ALL_IDS)
def test_plan_matches_oracle_workloads(grs, orc, cid):
    w = workloads.get(cid)
    op = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes)
    h = grs.grs_plan_create(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard,
                            w.bucket_bytes, grs.GRS_PLAN_HOST_ONLY)
    try:
        _compare_plan(grs, h, op, w.numels, w.owners)
    finally:
        grs.grs_plan_destroy(h)


GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "plan_layouts.json")))


@pytest.mark.parametrize("case", GOLD["cases"], ids=lambda c: c["name"])
def test_plan_matches_hand_layouts(grs, orc, case):
    h = grs.grs_plan_create_ex(case["numel"], case["owner"], case.get("tensor_flags"), case["world"],
                               case["tp"], case["dp_replicate"], case["dp_shard"], case["bucket_bytes"],
                               grs.GRS_PLAN_HOST_ONLY)
    try:
        op = oracle.plan(case["numel"], case["owner"], case["world"], case["tp"],
                         case["dp_replicate"], case["dp_shard"], case["bucket_bytes"],
                         case.get("tensor_flags"))
        _compare_plan(grs, h, op, case["numel"], case["owner"])
        info = grs.grs_plan_query(h)
        assert info["n_rank_pad"] == case["n_rank_pad"]
        assert info["n_state_pad"] == case["n_state_pad"]
    finally:
        grs.grs_plan_destroy(h)


@pytest.mark.parametrize("case", GOLD["rejections"], ids=lambda c: c["why"])
def test_plan_rejections_match(grs, case):
    with pytest.raises(grs.GrsError) as ei:
        grs.grs_plan_create_ex(case["numel"], case["owner"], case.get("tensor_flags"), case["world"],
                               case["tp"], case["dp_replicate"], case["dp_shard"], case["bucket_bytes"],
                               grs.GRS_PLAN_HOST_ONLY)
    assert ei.value.status == case["status"]
    assert grs.grs_last_error() != ""


def test_world_above_limit_rejected(grs):
    with pytest.raises(grs.GrsError) as ei:
        grs.grs_plan_create([8], [0], 256, 1, 1, 256, 64, grs.GRS_PLAN_HOST_ONLY)
    assert ei.value.status == grs.GRS_ERR_INVALID_ARG


def test_random_plans_match_oracle(grs, orc):
    rng = np.random.default_rng(1234)
    for trial in range(150):
        tp = int(rng.choice([1, 2, 3, 4]))
        dr = int(rng.choice([1, 2, 3]))
        ds = int(rng.choice([1, 2, 3, 4, 5]))
        n = int(rng.integers(1, 30))
        owners = [int(x) for x in rng.integers(0, 4, n)]
        numels = []
        for o in owners:
            k = int(rng.integers(0, 300))
            numels.append(k * tp if o == oracle.LOCAL_SHARD else k)
        bb = int(rng.choice([2, 16, 64, 250, 1000, 1 << 20]))
        world = tp * dr * ds
        dsa = -1 if rng.random() < 0.2 else ds
        flags = [int(x) for x in (rng.random(n) < 0.2)] if trial % 2 else None
        if flags is not None and all(flags):
            flags[0] = 0
        op = oracle.plan(numels, owners, world, tp, dr, dsa, bb, flags)
        h = grs.grs_plan_create_ex(numels, owners, flags, world, tp, dr, dsa, bb, grs.GRS_PLAN_HOST_ONLY)
        try:
            _compare_plan(grs, h, op, numels, owners)
        finally:
            grs.grs_plan_destroy(h)


def test_host_only_plan_refuses_launches(grs):
    h = grs.grs_plan_create([64], [0], 2, 1, 1, 2, 1 << 20, grs.GRS_PLAN_HOST_ONLY)
    try:
        assert grs.grs_plan_query(h)["device"] == -1
        with pytest.raises(grs.GrsError) as ei:
            grs.grs_reduce_all(h, [16, 16], 16, 0, 0, None, 0)
        assert ei.value.status == grs.GRS_ERR_NO_DEVICE
        with pytest.raises(grs.GrsError) as ei:
            hp = grs.make_adamw(1e-3, 0.9, 0.999, 1e-8, 0.0, 1.0, 1, 1)
            grs.grs_clip_adamw_step(h, hp, 16, 16, 16, 16, 16, 16, 0)
        assert ei.value.status == grs.GRS_ERR_NO_DEVICE
    finally:
        grs.grs_plan_destroy(h)


def test_query_bounds(grs):
    h = grs.grs_plan_create([64, 8], [0, 1], 1, 1, 1, 1, 1 << 20, grs.GRS_PLAN_HOST_ONLY)
    try:
        with pytest.raises(grs.GrsError):
            grs.grs_bucket_info(h, 2)
        with pytest.raises(grs.GrsError):
            grs.grs_tensor_info(h, -1)
    finally:
        grs.grs_plan_destroy(h)


def _host_plan(grs, w):
    return grs.grs_plan_create(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes,
                               grs.GRS_PLAN_HOST_ONLY)


def _check_shard_views(grs, plan, tp):
    """The shard views of one replica, (shard s, tp index t) for every s and
    t: each bucket's slice is shard_len elements of row t (LOCAL_SHARD) or
    row 0, with the valid elements of [s * shard_len, (s + 1) * shard_len);
    the views' norm-counted elements add up to the plan's unique elements
    (each counted once: LOCAL_SHARD rows by their own tp index, the other
    rows by tp index 0 only); out-of-range indices and views of views are
    refused."""
    info = grs.grs_plan_query(plan)
    nb = info["n_buckets"]
    bks = [grs.grs_bucket_info(plan, b) for b in range(nb)]
    total_unique = 0
    for t in range(tp):
        for s in range(info["dp_shard"]):
            v = grs.grs_plan_shard_view(plan, s, t)
            try:
                vi = grs.grs_plan_query(v)
                assert vi["n_buckets"] == nb and vi["n_rank_pad"] == 0 and vi["device"] == -1
                assert vi["n_state_pad"] == sum(int(b["shard_len"]) for b in bks)
                off, counted = 0, 0
                for b, pb in enumerate(bks):
                    vb = grs.grs_bucket_info(v, b)
                    L = int(pb["shard_len"])
                    used = max(0, min(L, int(pb["used"]) - s * L))
                    assert (vb["copies"], vb["padded"], vb["shard_len"], vb["used"], vb["state_offset"]) == \
                        (1, L, L, used, off)
                    assert vb["tag"] == pb["tag"]
                    if pb["tag"] == grs.GRS_LOCAL_SHARD or t == 0:
                        counted += used
                    off += L
                assert vi["n_unique"] == counted
                total_unique += vi["n_unique"]
                if nb:
                    with pytest.raises(grs.GrsError) as ei:
                        grs.grs_segment_info(v, 0, 0)
                    assert ei.value.status == grs.GRS_ERR_UNSUPPORTED_COMPOSITION
                with pytest.raises(grs.GrsError) as ei:
                    grs.grs_plan_shard_view(v, 0, 0)
                assert ei.value.status == grs.GRS_ERR_INVALID_ARG
            finally:
                grs.grs_plan_destroy(v)
    assert total_unique == info["n_unique"]
    for s, t in ((-1, 0), (info["dp_shard"], 0), (0, -1), (0, tp)):
        with pytest.raises(grs.GrsError) as ei:
            grs.grs_plan_shard_view(plan, s, t)
        assert ei.value.status == grs.GRS_ERR_INVALID_ARG


@pytest.mark.parametrize("cid", [0, 1, 3, 4])
def test_shard_views_partition_the_plan(grs, cid):
    """_check_shard_views on the workloads' plans."""
    w = workloads.get(cid)
    plan = _host_plan(grs, w)
    try:
        _check_shard_views(grs, plan, w.tp)
    finally:
        grs.grs_plan_destroy(plan)


def test_shard_views_partition_random_plans(grs):
    """_check_shard_views on random plans: every tag, frozen tensors,
    zero-size tensors, dp_shard = -1, bucket sizes from 2 bytes up."""
    rng = np.random.default_rng(4321)
    for trial in range(120):
        tp = int(rng.choice([1, 2, 3, 4]))
        dr = int(rng.choice([1, 2, 3]))
        ds = int(rng.choice([1, 2, 3, 4, 5, 8]))
        n = int(rng.integers(1, 30))
        owners = [int(x) for x in rng.integers(0, 4, n)]
        numels = [int(rng.integers(0, 300)) * (tp if o == oracle.LOCAL_SHARD else 1) for o in owners]
        flags = [int(x) for x in (rng.random(n) < 0.2)] if trial % 2 else None
        if flags is not None and all(flags):
            flags[0] = 0
        h = grs.grs_plan_create_ex(numels, owners, flags, tp * dr * ds, tp, dr,
                                   -1 if rng.random() < 0.2 else ds,
                                   int(rng.choice([2, 16, 64, 250, 1000, 1 << 20])), grs.GRS_PLAN_HOST_ONLY)
        try:
            _check_shard_views(grs, h, tp)
        finally:
            grs.grs_plan_destroy(h)
