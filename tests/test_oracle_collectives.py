"""Pin the oracle's reduction against real collectives on CPU ranks.

The pages validate multi-rank semantics with CPU reference checks (TP
replica ownership issue, "Preserved prototype and evidence": four-rank
CPU/NCCL reference checks).  Here world-size 4 and 8 gloo process groups
run the collectives the pages name, per owner tag, on each rank's own
bucket buffer:

  * TP:   all-reduce SUM over the TP group, then /tp for REPLICA_AVG
          (average across TP), kept as a sum for PARTIAL_SUM, skipped for
          LOCAL_SHARD (never synchronised as replicas) and ALREADY_REDUCED;
  * DP:   reduce-scatter SUM over the dp_shard group, all-reduce SUM across
          dp_replicate replicas, /dp (Cosmos 3 parallelism, section 2:
          all-reduce across replicas, shards hold 1/dp_shard), skipped for
          ALREADY_REDUCED (never reduced twice);
  * microbatches summed.

Each rank's shard, and the all-gathered bucket, must equal the oracle's.
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from oracle import ALREADY_REDUCED, LOCAL_SHARD, PARTIAL_SUM, REPLICA_AVG


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _bits_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _worker(rank, world, port, path, tp, dr, ds):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = np.load(path)
        t = rank % tp
        s = (rank // tp) % ds
        r = rank // (tp * ds)
        # groups: every rank creates every group, in the same order
        tp_groups, shard_groups, rep_groups = {}, {}, {}
        for rr in range(dr):
            for ss in range(ds):
                tp_groups[(rr, ss)] = dist.new_group([oracle.rank(rr, ss, x, ds, tp) for x in range(tp)])
        for rr in range(dr):
            for tt in range(tp):
                shard_groups[(rr, tt)] = dist.new_group([oracle.rank(rr, x, tt, ds, tp) for x in range(ds)])
        for ss in range(ds):
            for tt in range(tp):
                rep_groups[(ss, tt)] = dist.new_group([oracle.rank(x, ss, tt, ds, tp) for x in range(dr)])
        tpg, shg, rpg = tp_groups[(r, s)], shard_groups[(r, t)], rep_groups[(s, t)]
        dp = dr * ds
        nb = int(d["n_buckets"])
        for b in range(nb):
            tag = int(d["b_tag"][b])
            P = int(d["b_padded"][b])
            used = int(d["b_used"][b])
            L = P // ds
            grads = d[f"grads{b}"]  # [M][R][P]
            M = grads.shape[0]
            shard_acc = torch.zeros(L, dtype=torch.float64)
            for j in range(M):
                x = torch.tensor(_bits_to_f64(grads[j, rank]))
                x[used:] = 0.0  # collectives carry no padding garbage
                if tag == ALREADY_REDUCED:
                    shard_acc += x[s * L:(s + 1) * L]
                    continue
                if tag in (REPLICA_AVG, PARTIAL_SUM) and tp > 1:
                    dist.all_reduce(x, op=dist.ReduceOp.SUM, group=tpg)
                if tag == REPLICA_AVG:
                    x /= tp
                out = torch.zeros(L, dtype=torch.float64)
                if ds > 1:
                    dist.reduce_scatter(out, list(x.split(L)), op=dist.ReduceOp.SUM, group=shg)
                else:
                    out.copy_(x)
                if dr > 1:
                    dist.all_reduce(out, op=dist.ReduceOp.SUM, group=rpg)
                shard_acc += out / dp
            copy = t if tag == LOCAL_SHARD else 0
            want = d[f"acc{b}"][copy]
            np.testing.assert_allclose(shard_acc.numpy(), want[s * L:(s + 1) * L], rtol=1e-12, atol=1e-18)
            full = [torch.zeros(L, dtype=torch.float64) for _ in range(ds)]
            if ds > 1:
                dist.all_gather(full, shard_acc, group=shg)
            else:
                full = [shard_acc]
            np.testing.assert_allclose(torch.cat(full).numpy(), want, rtol=1e-12, atol=1e-18)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("tp,dr,ds", [(2, 1, 2), (2, 2, 2), (1, 2, 2)])
def test_oracle_matches_gloo_collectives(orc, tp, dr, ds):
    rng = np.random.default_rng(100 + tp * 10 + dr * 3 + ds)
    world = tp * dr * ds
    M = 2
    numels = [21, 5, 18, 3, 40, 12]
    owners = [REPLICA_AVG, PARTIAL_SUM, LOCAL_SHARD, ALREADY_REDUCED, REPLICA_AVG, LOCAL_SHARD]
    numels = [n if o != LOCAL_SHARD else n - n % tp for n, o in zip(numels, owners)]
    p = oracle.plan(numels, owners, world, tp, dr, ds, 64)
    arrays = {"n_buckets": np.int64(p.n_buckets), "b_tag": p.b_tag, "b_padded": p.b_padded,
              "b_used": p.b_used}
    for b in range(p.n_buckets):
        P = int(p.b_padded[b])
        used = int(p.b_used[b])
        vals = rng.normal(0, 1e-2, (M, world, P)).astype(np.float32)
        bits = torch.tensor(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
        if int(p.b_tag[b]) == ALREADY_REDUCED:
            bits[:, :, :] = bits[:, :1, :]  # an already-reduced gradient is the same everywhere
        oracle_in = bits.copy()
        oracle_in[:, :, used:] = 0x7FC0  # NaN padding: the oracle must mask it
        arrays[f"grads{b}"] = bits
        arrays[f"acc{b}"] = oracle.reduce_bucket(int(p.b_tag[b]), tp, dr, ds, P, used, oracle_in)
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "case.npz")
        np.savez(path, **arrays)
        mp.start_processes(_worker, args=(world, _free_port(), path, tp, dr, ds), nprocs=world,
                           start_method="spawn", join=True)


# ---------------------------------------------------------------------------
# The whole sharded step across real ranks: after the reduce-scatter (and
# the all-reduce across replicas), each rank (r, s, t) owns shard s of its
# bucket rows.  It adds its shard's share of the global squared norm (every
# unique element once: replica 0 only, tp index 0 only for tensors that are
# the same on every tp rank), one scalar all-reduce gives the norm, the rank
# runs clip + AdamW on its shard alone, and an all-gather of the bf16 shards
# over the shard group rebuilds the full parameters ("Cosmos 3 ...
# distributed parallelism", section 2: all-reduce across replicas, all-gather
# across shards).  The result must equal the single-process oracle's update
# of the whole bucket layout: the layout this library keeps in one GPU's
# memory is that decomposition's.
# ---------------------------------------------------------------------------
def _f32_ulps(a, b):
    a = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    a = np.where(a < 0, -(a & 0x7FFFFFFF), a)
    b = np.where(b < 0, -(b & 0x7FFFFFFF), b)
    return np.abs(a - b)


def _step_worker(rank, world, port, path, tp, dr, ds):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = np.load(path)
        t = rank % tp
        s = (rank // tp) % ds
        r = rank // (tp * ds)
        tp_groups, shard_groups, rep_groups = {}, {}, {}
        for rr in range(dr):
            for ss in range(ds):
                tp_groups[(rr, ss)] = dist.new_group([oracle.rank(rr, ss, x, ds, tp) for x in range(tp)])
        for rr in range(dr):
            for tt in range(tp):
                shard_groups[(rr, tt)] = dist.new_group([oracle.rank(rr, x, tt, ds, tp) for x in range(ds)])
        for ss in range(ds):
            for tt in range(tp):
                rep_groups[(ss, tt)] = dist.new_group([oracle.rank(x, ss, tt, ds, tp) for x in range(dr)])
        tpg, shg, rpg = tp_groups[(r, s)], shard_groups[(r, t)], rep_groups[(s, t)]
        dp = dr * ds
        nb = int(d["n_buckets"])
        hp = tuple(float(x) for x in d["hp"])
        max_norm = float(d["max_norm"])
        shards = []
        local_sq = 0.0
        for b in range(nb):
            tag = int(d["b_tag"][b])
            P = int(d["b_padded"][b])
            used = int(d["b_used"][b])
            L = P // ds
            grads = d[f"grads{b}"]
            M = grads.shape[0]
            shard_acc = torch.zeros(L, dtype=torch.float64)
            for j in range(M):
                x = torch.tensor(_bits_to_f64(grads[j, rank]))
                x[used:] = 0.0
                if tag == ALREADY_REDUCED:
                    shard_acc += x[s * L:(s + 1) * L]
                    continue
                if tag in (REPLICA_AVG, PARTIAL_SUM) and tp > 1:
                    dist.all_reduce(x, op=dist.ReduceOp.SUM, group=tpg)
                if tag == REPLICA_AVG:
                    x /= tp
                out = torch.zeros(L, dtype=torch.float64)
                if ds > 1:
                    dist.reduce_scatter(out, list(x.split(L)), op=dist.ReduceOp.SUM, group=shg)
                else:
                    out.copy_(x)
                if dr > 1:
                    dist.all_reduce(out, op=dist.ReduceOp.SUM, group=rpg)
                shard_acc += out / dp
            row = t if tag == LOCAL_SHARD else 0
            n_used = max(0, min(L, used - s * L))
            a = shard_acc.numpy()
            owner_of_unique = r == 0 and (tag == LOCAL_SHARD or t == 0)
            if owner_of_unique:
                local_sq += oracle.norm_sq(a[:n_used], M)
            shards.append((b, row, L, n_used, a, M))
        # the library's shard view of this rank describes the same slices
        if "numels" in d.files:
            from gradient_reduction_sharded_gb300 import grs
            plan = grs.grs_plan_create([int(x) for x in d["numels"]], [int(x) for x in d["owners"]], world, tp, dr,
                                       ds, int(d["bucket_bytes"]), grs.GRS_PLAN_HOST_ONLY)
            view = grs.grs_plan_shard_view(plan, s, t)
            try:
                off = 0
                for b, row, L, n_used, a, M in shards:
                    vb = grs.grs_bucket_info(view, b)
                    assert (vb["state_offset"], vb["padded"], vb["used"]) == (off, L, n_used), (rank, b)
                    off += L
                counted = sum(n_used for b, row, L, n_used, a, M in shards
                              if int(d["b_tag"][b]) == LOCAL_SHARD or t == 0)
                assert grs.grs_plan_query(view)["n_unique"] == counted
            finally:
                grs.grs_plan_destroy(view)
                grs.grs_plan_destroy(plan)
        S = torch.tensor([local_sq], dtype=torch.float64)
        dist.all_reduce(S, op=dist.ReduceOp.SUM)  # the one scalar exchange of the norm
        S = float(S[0])
        np.testing.assert_allclose(S, float(d["norm_sq"]), rtol=1e-12)
        c = oracle.clip_coef(S, max_norm)
        for b, row, L, n_used, a, M in shards:
            o = int(d["b_state_off"][b]) + row * int(d["b_padded"][b]) + s * L
            m0 = np.zeros(L, np.float32)
            p1, m1, v1, bits = oracle.adamw(a, n_used, M, c, hp, 1, d["master0"][o:o + L], m0, m0)
            for got, want, what in ((p1, d["master1"][o:o + L], "master"), (m1, d["m1"][o:o + L], "m"),
                                    (v1, d["v1"][o:o + L], "v")):
                assert _f32_ulps(got, want).max() <= 1, (b, what)
            # all-gather of the bf16 shards over the shard group -> the row
            mine = torch.tensor(bits.astype(np.int32))
            full = [torch.zeros(L, dtype=torch.int32) for _ in range(ds)]
            if ds > 1:
                dist.all_gather(full, mine, group=shg)
            else:
                full = [mine]
            row_bits = torch.cat(full).numpy().astype(np.uint16)
            P = int(d["b_padded"][b])
            want_row = d["bits1"][o - s * L:o - s * L + P]
            diff = np.abs(row_bits.view(np.int16).astype(np.int64) - want_row.view(np.int16).astype(np.int64))
            assert diff.max() <= 1, b
            # every replica holds the same shard after the step
            if dr > 1:
                reps = [torch.zeros(L, dtype=torch.float32) for _ in range(dr)]
                dist.all_gather(reps, torch.tensor(p1), group=rpg)
                assert all(torch.equal(reps[0], x) for x in reps)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("tp,dr,ds", [(2, 1, 2), (1, 2, 2), (2, 2, 2)])
def test_sharded_step_matches_single_process_oracle(orc, tp, dr, ds):
    from gradient_reduction_sharded_gb300 import _build
    _build.build()  # the ranks also check the library's shard views (host tables only)
    rng = np.random.default_rng(300 + tp * 10 + dr * 3 + ds)
    world = tp * dr * ds
    M = 2
    numels = [21, 5, 18, 3, 40, 12, 37]
    owners = [REPLICA_AVG, PARTIAL_SUM, LOCAL_SHARD, ALREADY_REDUCED, REPLICA_AVG, LOCAL_SHARD, PARTIAL_SUM]
    numels = [n if o != LOCAL_SHARD else n - n % tp for n, o in zip(numels, owners)]
    p = oracle.plan(numels, owners, world, tp, dr, ds, 64)
    hp = (1e-3, 0.9, 0.999, 1e-8, 0.01)
    max_norm = 0.01  # clipping active
    arrays = {"n_buckets": np.int64(p.n_buckets), "b_tag": p.b_tag, "b_padded": p.b_padded,
              "b_used": p.b_used, "b_state_off": p.b_state_off, "hp": np.array(hp), "max_norm": max_norm,
              "numels": np.array(numels), "owners": np.array(owners), "bucket_bytes": np.int64(64)}
    inputs = {}
    for b in range(p.n_buckets):
        P = int(p.b_padded[b])
        vals = rng.normal(0, 1e-2, (M, world, P)).astype(np.float32)
        bits = torch.tensor(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
        if int(p.b_tag[b]) == ALREADY_REDUCED:
            bits[:, :, :] = bits[:, :1, :]
        inputs[b] = bits
        arrays[f"grads{b}"] = bits
    master0 = rng.normal(0, 0.02, p.n_state_pad).astype(np.float32)
    z = np.zeros(p.n_state_pad, np.float32)
    res = oracle.full_update(p, lambda b: inputs[b], M, hp, max_norm, 1, master0, z, z)
    assert res.clip < 1.0
    arrays.update(norm_sq=res.norm_sq, master0=master0, master1=res.master, m1=res.m, v1=res.v,
                  bits1=res.params_bf16)
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "case.npz")
        np.savez(path, **arrays)
        mp.start_processes(_step_worker, args=(world, _free_port(), path, tp, dr, ds), nprocs=world,
                           start_method="spawn", join=True)
