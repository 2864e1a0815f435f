"""Checkpoint, restore and reshard on the GPU.

A run under geometry A (world 16: tp 2, dp_replicate 2, dp_shard 4) takes
one update and is saved; the checkpoint is restored under geometry B (the
same 16 ranks as dp_replicate 4 x dp_shard 2, or another bucket size and an
ownership change).  The restored state equals the saved one element for
element in the canonical logical order (checked with the oracle's own layout
conversion), and the next update from the restored state equals the
uninterrupted run's next update.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_support import Case, Run, grs

pytestmark = pytest.mark.gpu

RA, PS, LS, AR = 0, 1, 2, 3
NUMELS = [100003, 1024, 65536 * 2, 4099, 333, 70001, 8000]
OWNERS = [RA, PS, LS, AR, PS, RA, LS]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.init()


def spec_of(ck, c: Case):
    return ck.PlanSpec(c.numels, c.owners, c.tensor_flags, c.world, c.tp, c.dp_replicate, c.dp_shard,
                       c.bucket_bytes, 0)


def relayout_grads(src: Run, dst: Run):
    """Give `dst` the same per-rank, per-tensor gradients as `src` (test input
    preparation: each rank's tensor slices copied between the two layouts)."""
    a, b = src.op, dst.op
    for j in range(src.c.n_micro):
        for k in range(src.c.world):
            dst.grads[j][k].zero_()
            for i in range(len(a.numel)):
                ba, bb = int(a.t_bucket[i]), int(b.t_bucket[i])
                if ba < 0 or bb < 0:
                    continue
                n = a.per_rank(i)
                oa = int(a.b_rank_off[ba]) + int(a.t_offset[i])
                ob = int(b.b_rank_off[bb]) + int(b.t_offset[i])
                dst.grads[j][k][ob:ob + n] = src.grads[j][k][oa:oa + n]


def logical(run: Run, t: torch.Tensor) -> np.ndarray:
    return oracle.to_logical(run.op, t[:run.nsp].cpu().numpy())


def test_restore_reshard_and_continue(tmp_path):
    from gradient_reduction_sharded_gb300 import checkpoint as ck
    ca = Case(NUMELS, OWNERS, 16, 2, 2, 4, 1 << 18, 2, 1e-3, 51)
    cb = Case(NUMELS, OWNERS, 16, 2, 4, 2, 1 << 18, 2, 1e-3, 51)
    a, b = Run(ca), Run(cb)
    try:
        a.update()
        torch.cuda.synchronize()
        d = str(tmp_path / "ckpt")
        ck.save(d, a.plan, spec_of(ck, ca), {"master": a.master, "exp_avg": a.m, "exp_avg_sq": a.v},
                {"step": 1})
        man = ck.load(d, b.plan, {"master": b.master, "exp_avg": b.m, "exp_avg_sq": b.v})
        assert man["steps"] == {"step": 1}
        for ta, tb in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert np.array_equal(logical(a, ta), logical(b, tb))
        # padding of the reader's layout is exactly zero
        pad = np.ones(b.nsp, bool)
        for bb in range(b.op.n_buckets):
            for t in range(b.op.copies(bb)):
                o = int(b.op.b_state_off[bb]) + t * int(b.op.b_padded[bb])
                pad[o:o + int(b.op.b_used[bb])] = False
        assert np.all(b.master[:b.nsp].cpu().numpy()[pad] == 0)
        # continue: the same logical gradients on both, step 2
        a.fill_grads(step_seed=2)
        relayout_grads(a, b)
        b.step = 1
        a.update()
        b.update()
        torch.cuda.synchronize()
        for ta, tb in ((a.acc, b.acc), (a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert np.array_equal(logical(a, ta), logical(b, tb))
        assert float(a.norm.cpu()[0]) == float(b.norm.cpu()[0])
    finally:
        a.close()
        b.close()


def test_restore_across_bucket_size_and_ownership(tmp_path):
    """Legacy ownership -> native ownership: the same logical parameters
    with another owner tag on two tensors and another bucket size restore
    exactly (the state does not depend on how gradients are reduced)."""
    from gradient_reduction_sharded_gb300 import checkpoint as ck
    ca = Case(NUMELS, OWNERS, 8, 2, 1, 4, 1 << 18, 1, 1e-3, 52)
    owners_b = list(OWNERS)
    owners_b[1] = RA   # a norm vector: partial sums -> replica average
    owners_b[6] = RA   # a TP-sharded tensor -> replicated
    cb = Case(NUMELS, owners_b, 8, 2, 1, 4, 1 << 14, 1, 1e-3, 52)
    a, b = Run(ca), Run(cb)
    try:
        a.update()
        torch.cuda.synchronize()
        d = str(tmp_path / "ckpt2")
        saving = ck.save_async(d, a.plan, spec_of(ck, ca), {"master": a.master, "exp_avg": a.m,
                                                            "exp_avg_sq": a.v}, {"step": 1})
        saving.wait()
        ck.load(d, b.plan, {"master": b.master, "exp_avg": b.m, "exp_avg_sq": b.v})
        for ta, tb in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert np.array_equal(logical(a, ta), logical(b, tb))
    finally:
        a.close()
        b.close()


def test_restore_many_small_tensors_across_tp(tmp_path):
    """1500 small tensors of all tags (zero-size and frozen ones among them)
    saved under tp 2 x dp_replicate 2 x dp_shard 4 and restored under tp 4 x
    dp_shard 4 with another bucket size: the logical state is identical and
    every padding element of the reader's layout is zero."""
    from gradient_reduction_sharded_gb300 import checkpoint as ck
    rng = np.random.default_rng(31)
    owners = rng.integers(0, 4, 1500).tolist()
    numels = [int(x) * (4 if o == LS else 1) for x, o in zip(rng.integers(0, 120, 1500), owners)]
    flags = [1 if i % 97 == 5 else 0 for i in range(1500)]
    ca = Case(numels, owners, 16, 2, 2, 4, 1 << 15, 1, 1e-2, 54, tensor_flags=flags)
    cb = Case(numels, owners, 16, 4, 1, 4, 1 << 13, 1, 1e-2, 54, tensor_flags=flags)
    a, b = Run(ca), Run(cb)
    try:
        a.update()
        torch.cuda.synchronize()
        d = str(tmp_path / "ckpt3")
        ck.save(d, a.plan, spec_of(ck, ca), {"master": a.master, "exp_avg": a.m, "exp_avg_sq": a.v},
                {"step": 1})
        for t in (b.master, b.m, b.v):
            t.fill_(float("nan"))
        ck.load(d, b.plan, {"master": b.master, "exp_avg": b.m, "exp_avg_sq": b.v})
        pad = np.ones(b.nsp, bool)
        for bb in range(b.op.n_buckets):
            for t in range(b.op.copies(bb)):
                o = int(b.op.b_state_off[bb]) + t * int(b.op.b_padded[bb])
                pad[o:o + int(b.op.b_used[bb])] = False
        for ta, tb in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert np.array_equal(logical(a, ta), logical(b, tb))
            hb = tb[:b.nsp].cpu().numpy()
            assert np.all(hb[pad] == 0) and not np.isnan(hb).any()
    finally:
        a.close()
        b.close()


def test_state_logical_kernels_match_oracle():
    c = Case([21, 5, 18, 3, 1001, 77, 4096], [RA, PS, LS, AR, RA, PS, LS], 6, 2, 1, 3, 256, 1, 1e-2, 53,
             tensor_flags=[0, 0, 0, 1, 0, 0, 0])
    run = Run(c)
    try:
        g = grs()
        info = run.info
        gen = torch.Generator(device="cuda").manual_seed(9)
        st = torch.randn(run.nsp, generator=gen, device="cuda")
        lg = torch.empty(info["n_unique"], device="cuda")
        g.grs_state_to_logical(run.plan, st.data_ptr(), lg.data_ptr(), run.stream())
        torch.cuda.synchronize()
        want = oracle.to_logical(run.op, st.cpu().numpy())
        assert np.array_equal(lg.cpu().numpy(), want)
        back = torch.full((run.nsp,), 5.0, device="cuda")
        g.grs_state_from_logical(run.plan, lg.data_ptr(), back.data_ptr(), run.stream())
        torch.cuda.synchronize()
        assert np.array_equal(back.cpu().numpy(), oracle.from_logical(run.op, want))
    finally:
        run.close()
