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
