"""The bench's byte accounting (the roofline's numerator), on the CPU.

The per-update mandatory bytes of the five workloads against the figures
stated for them independently of this code (per unique padded element:
2*M*R_e + 4 + 8*(M-1) + 30, summed over the buckets of each plan), and the
variant accounting (fp32 gradients, tensors without a gradient) against
counts done by hand on the tiny plan.
"""
import pytest

import bench
import workloads

# GB (1e9 bytes) per update, from the scope table of the hot path.
STATED_GB = {1: 4.16, 2: 239.8, 3: 196.8, 4: 134.9}


@pytest.mark.parametrize("cid", sorted(STATED_GB))
def test_mandatory_bytes_match_stated_totals(cid):
    w = workloads.get(cid)
    op = bench._oracle_plan(w)
    mb = bench.mandatory_bytes(bench.oracle_buckets(op), w.n_micro)
    assert round(mb["total"] / 1e9, 1 if cid > 1 else 2) == STATED_GB[cid]
    assert mb["update"] == 30 * op.n_state_pad


def test_tiny_plan_bytes_by_hand():
    # tiny plan (world 4, tp 2, dp_shard 2, dp 2): buckets RA [64x64 + 256x64
    # = 20480], PS [32], LS [(128x64 + 64x128)/2 = 8192 per row, 2 rows],
    # AR [64]; padded to multiples of 16: 20480, 32, 8192, 64.
    w = workloads.get(0)
    op = bench._oracle_plan(w)
    geo = bench.oracle_buckets(op)
    assert [(g["tag"], g["copies"], g["padded"], g["group_size"]) for g in geo] == [
        (0, 1, 20480, 4), (1, 1, 32, 4), (2, 2, 8192, 2), (3, 1, 64, 1)]
    red = 20480 * (2 * 4 + 4) + 32 * (2 * 4 + 4) + 2 * 8192 * (2 * 2 + 4) + 64 * (2 * 1 + 4)
    mb = bench.mandatory_bytes(geo, 1)
    assert mb["reduce"] == red
    assert mb["update"] == 30 * (20480 + 32 + 2 * 8192 + 64)
    # fp32 gradients: 4 bytes per rank element read
    red32 = 20480 * (4 * 4 + 4) + 32 * (4 * 4 + 4) + 2 * 8192 * (4 * 2 + 4) + 64 * (4 * 1 + 4)
    assert bench.mandatory_bytes(geo, 1, 4)["reduce"] == red32
    # two microbatches: the second reads and writes the accumulator (8 more)
    red2 = 20480 * (2 * 2 * 4 + 4 + 8) + 32 * (2 * 2 * 4 + 12) + 2 * 8192 * (2 * 2 * 2 + 12) + 64 * (2 * 2 + 12)
    assert bench.mandatory_bytes(geo, 2)["reduce"] == red2


def test_unused_variant_bytes_by_hand():
    w = workloads.get(0)
    op = bench._oracle_plan(w)
    used = bench.unused_pattern(len(w.numels))
    assert used == [1, 1, 1, 0, 1, 1]  # the AR bias b[64] has no gradient
    idle = 64
    n_unique = sum(w.numels)
    vb = bench.variant_bytes(bench.oracle_buckets(op), 1, 2, op.n_state_pad, n_unique, idle)
    assert vb["norm"] == 0  # fused into the masked reduction
    assert vb["norm_pass"] == 4 * (n_unique - 64)
    assert vb["update"] == 30 * (op.n_state_pad - 64)
    assert vb["total"] == vb["reduce"] + vb["norm"] + vb["update"]
    plain = bench.variant_bytes(bench.oracle_buckets(op), 1, 2, op.n_state_pad, n_unique)
    assert plain["norm"] == 0 and plain["total"] == plain["reduce"] + plain["update"]


def test_frozen_pattern_leaves_the_plan_smaller():
    w = workloads.get(1)
    flags = bench.frozen_pattern(len(w.numels))
    assert sum(flags) == 20 and flags[:20] == [1] * 20
    op = bench._oracle_plan(w, flags)
    assert sum(n for n, f in zip(w.numels, flags) if not f) == 50343936
    assert op.n_state_pad >= 50343936


def test_e2e_pinned_host_bytes():
    """The end-to-end leg pins every rank's gradients of every microbatch
    and the bf16 parameters: 2 bytes per element of each."""
    import types
    import bench
    u = types.SimpleNamespace(n_micro=3, w=types.SimpleNamespace(world=4),
                              info={"n_rank_pad": 1000, "n_state_pad": 700})
    assert bench.e2e_host_bytes(u) == (3 * 4 * 1000 + 700) * 2
    avail = bench.host_available_bytes()
    assert avail is None or avail > 0


def test_profiling_slices_keep_the_geometry():
    """The one-layer slices that stand in for the 1.1B, MoE and 3.2B plans in
    ncu captures keep the degrees, microbatches, owner tags and per-layer
    tensor shapes, and are small (under 130M parameters)."""
    import workloads
    for cid in (2, 3, 4):
        full, sl = workloads.get(cid), workloads.get(cid, layers=1)
        for k in ("tp", "dp_replicate", "dp_shard", "world", "n_micro", "bucket_bytes", "grad_std"):
            assert getattr(full, k) == getattr(sl, k), (cid, k)
        assert sl.n_unique < 130_000_000 < full.n_unique
        assert set(sl.owners) == set(full.owners)
        layer0 = [(t.name, t.shape, t.owner) for t in full.tensors if t.name.startswith("layers.0.")]
        sl0 = [(t.name, t.shape, t.owner) for t in sl.tensors if t.name.startswith("layers.0.")]
        if cid == 3:  # the MoE slice keeps 8 of the 32 experts (and the router's 8 outputs)
            layer0 = [(n, ((8,) + s[1:]) if "experts" in n else (s[0], 8) if n.endswith("router") else s, o)
                      for n, s, o in layer0]
        assert layer0 == sl0, cid
        assert not any(t.name.startswith("layers.1.") for t in sl.tensors)
    with __import__("pytest").raises(ValueError):
        workloads.get(1, layers=1)
