"""The benchmark's multi-rank host logic on CPU gloo ranks (world size 2):
the step time reported is the slowest rank's, and the whole-job value counts
every replica's update."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks(1.5 + rank, "cpu")
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value():
    import bench
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, _port(), out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == out[1] == 2.5
    assert bench.job_value(2.5, 2) == 1.25
    assert bench.max_over_ranks(3.0) == 3.0  # no process group: identity


def test_gpus_flag_launches_one_rank_per_gpu():
    """bench.py --gpus N outside torchrun re-launches itself as N ranks on
    one node, rendezvous on 127.0.0.1, with the same arguments."""
    import bench
    cmd = bench.rank_launch_cmd(4, ["--gpus", "4", "--steps", "7"], 29555)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--nnodes=1" in cmd
    i = cmd.index("--master-addr")
    assert cmd[i + 1] == "127.0.0.1" and cmd[cmd.index("--master-port") + 1] == "29555"
    assert cmd[-4:] == ["--gpus", "4", "--steps", "7"] and cmd[-5].endswith("bench.py")
