"""Pins of the CPU oracle against values that the pages or mathematics fix.

Each test ties one oracle function to something other than the oracle:
hand-checked values (tests/golden), closed forms, invariants of the owner
semantics, torch.optim.AdamW, torch.nn.utils.clip_grad_norm_ and torch's
bf16 cast.  A plausible slip in the oracle (a dropped term, a wrong scale,
a swapped mesh index) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import ALREADY_REDUCED, LOCAL_SHARD, PARTIAL_SUM, REPLICA_AVG

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TAGS = {"REPLICA_AVG": REPLICA_AVG, "PARTIAL_SUM": PARTIAL_SUM,
        "LOCAL_SHARD": LOCAL_SHARD, "ALREADY_REDUCED": ALREADY_REDUCED}


def bf16(x):
    """float values -> bf16 bit patterns (torch's round-to-nearest-even)."""
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Owner semantics, hand-checked (golden/hand_checked_world4.json)
# --------------------------------------------------------------------------
def test_hand_checked_single_microbatch(orc):
    g = load("hand_checked_world4.json")
    geo = g["geometry"]
    vals = g["rank_values"]
    P = 16
    grads = np.zeros((1, 4, P), np.uint16)
    for k, v in enumerate(vals):
        grads[0, k, :] = bf16([v] * P)
    for name, exp in g["expected_acc"].items():
        acc = oracle.reduce_bucket(TAGS[name], geo["tp"], geo["dp_replicate"], geo["dp_shard"],
                                   P, P, grads)
        assert acc.shape[0] == len(exp)
        for c, row in enumerate(exp):
            assert np.all(acc[c] == row[0]), (name, c, acc[c][:4], row)


def test_hand_checked_two_microbatches(orc):
    g = load("hand_checked_world4.json")["two_microbatch_case"]
    geo = g["geometry"]
    P = 8
    grads = np.zeros((2, 4, P), np.uint16)
    for j, vals in enumerate(g["rank_values_per_microbatch"]):
        for k, v in enumerate(vals):
            grads[j, k, :] = bf16([v] * P)
    for name, exp in g["expected_acc"].items():
        acc = oracle.reduce_bucket(TAGS[name], geo["tp"], geo["dp_replicate"], geo["dp_shard"],
                                   P, P, grads)
        for c, row in enumerate(exp):
            assert np.all(acc[c] == row[0]), (name, c, acc[c][:4], row)
        # G = acc / M: the norm of a constant bucket is P * (acc/M)^2
        s = oracle.norm_sq(acc, 2)
        want = sum(P * (row[0] / 2) ** 2 for row in exp)
        assert s == want


def test_hand_checked_fp32_gradients(orc):
    """The same hand-checked values through the fp32-gradient entry."""
    g = load("hand_checked_world4.json")
    geo = g["geometry"]
    P = 16
    grads = np.zeros((1, 4, P), np.float32)
    for k, v in enumerate(g["rank_values"]):
        grads[0, k, :] = v
    for name, exp in g["expected_acc"].items():
        acc = oracle.reduce_bucket(TAGS[name], geo["tp"], geo["dp_replicate"], geo["dp_shard"],
                                   P, P, grads)
        for c, row in enumerate(exp):
            assert np.all(acc[c] == row[0]), (name, c)


@pytest.mark.parametrize("tag", [REPLICA_AVG, PARTIAL_SUM, LOCAL_SHARD, ALREADY_REDUCED])
def test_fp32_and_bf16_entries_agree_on_bf16_values(orc, tag):
    """fp32 inputs that are exactly bf16 values reduce to the same result as
    the bf16 entry (the two decodings cannot disagree)."""
    rng = np.random.default_rng(12)
    tp, dr, ds, M, P = 2, 2, 2, 3, 40
    bits = bf16(rng.normal(0, 1e-2, (M, tp * dr * ds, P)))
    a = oracle.reduce_bucket(tag, tp, dr, ds, P, 33, bits)
    b = oracle.reduce_bucket(tag, tp, dr, ds, P, 33, bits_to_f32(bits).reshape(bits.shape))
    assert np.array_equal(a, b)


def test_dp_mesh_rank_order(orc):
    g = load("hand_checked_world4.json")["dp_mesh_2x4"]
    geo = g["geometry"]
    for r, row in enumerate(g["ranks"]):
        for s, want in enumerate(row):
            assert oracle.rank(r, s, 0, geo["dp_shard"], geo["tp"]) == want


def test_padding_ignored_and_zero(orc):
    """Input padding may hold NaN; outputs there are exactly zero."""
    P, used = 16, 5
    grads = np.full((2, 4, P), 0x7FC0, np.uint16)  # NaN everywhere
    grads[:, :, :used] = bf16(np.arange(1, used + 1))
    for tag in range(4):
        acc = oracle.reduce_bucket(tag, 2, 1, 2, P, used, grads)
        assert np.all(np.isfinite(acc))
        assert np.all(acc[:, used:] == 0.0)


# --------------------------------------------------------------------------
# Identical copies x: RA -> x, PS -> tp*x, LS -> x, AR -> x (per microbatch)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("tp,dr,ds", [(2, 1, 2), (2, 2, 4), (4, 1, 2), (1, 2, 4), (3, 1, 3)])
def test_identical_copies(orc, tp, dr, ds):
    rng = np.random.default_rng(7)
    R, P = tp * dr * ds, 40
    x = bf16(rng.normal(0, 1e-2, P))
    xv = bits_to_f32(x).astype(np.float64)
    grads = np.broadcast_to(x, (1, R, P)).copy()
    exp = {REPLICA_AVG: xv, PARTIAL_SUM: tp * xv, LOCAL_SHARD: xv, ALREADY_REDUCED: xv}
    for tag, want in exp.items():
        acc = oracle.reduce_bucket(tag, tp, dr, ds, P, P, grads)
        for c in range(acc.shape[0]):
            np.testing.assert_allclose(acc[c], want, rtol=1e-15, atol=0)


# --------------------------------------------------------------------------
# No double reduction, no TP sync of local shards
# --------------------------------------------------------------------------
def test_already_reduced_ignores_other_ranks(orc):
    rng = np.random.default_rng(1)
    tp, dr, ds, P = 2, 2, 2, 24
    R = tp * dr * ds
    grads = bf16(rng.normal(0, 1, (2, R, P)))
    base = oracle.reduce_bucket(ALREADY_REDUCED, tp, dr, ds, P, P, grads)
    pert = grads.copy()
    pert[:, 1:, :] = bf16(rng.normal(0, 5, (2, R - 1, P)))
    again = oracle.reduce_bucket(ALREADY_REDUCED, tp, dr, ds, P, P, pert)
    assert np.array_equal(base, again)
    # ... and rank 0's copy is what it returns, summed over microbatches
    want = bits_to_f32(grads[0, 0]).astype(np.float64) + bits_to_f32(grads[1, 0])
    assert np.array_equal(base[0], want)


def test_local_shard_not_synchronised_across_tp(orc):
    rng = np.random.default_rng(2)
    tp, dr, ds, P = 2, 2, 2, 24
    R = tp * dr * ds
    grads = bf16(rng.normal(0, 1, (1, R, P)))
    base = oracle.reduce_bucket(LOCAL_SHARD, tp, dr, ds, P, P, grads)
    for tprime in range(tp):
        pert = grads.copy()
        for r in range(dr):
            for s in range(ds):
                k = oracle.rank(r, s, tprime, ds, tp)
                pert[0, k] = bf16(rng.normal(0, 3, P))
        again = oracle.reduce_bucket(LOCAL_SHARD, tp, dr, ds, P, P, pert)
        for t in range(tp):
            if t == tprime:
                assert not np.array_equal(base[t], again[t])
            else:
                assert np.array_equal(base[t], again[t])


def test_partial_sum_is_a_sum_not_the_local_value(orc):
    """The Megatron-FSDP bug class on the issue page: copying the local grad
    without resolving a TP Partial placement loses the sum."""
    tp, dr, ds, P = 2, 1, 1, 8
    grads = np.zeros((1, 2, P), np.uint16)
    grads[0, 0] = bf16([1.0] * P)
    grads[0, 1] = bf16([2.0] * P)
    acc = oracle.reduce_bucket(PARTIAL_SUM, tp, dr, ds, P, P, grads)
    assert np.all(acc[0] == 3.0)
    acc = oracle.reduce_bucket(REPLICA_AVG, tp, dr, ds, P, P, grads)
    assert np.all(acc[0] == 1.5)


# --------------------------------------------------------------------------
# Accumulation equals one large batch
# --------------------------------------------------------------------------
@pytest.mark.parametrize("tag", [REPLICA_AVG, PARTIAL_SUM, LOCAL_SHARD])
def test_accumulation_equals_large_batch(orc, tag):
    """M microbatches over dp ranks give the same G as one microbatch over a
    world whose replica axis is M times larger (mean of means = mean)."""
    rng = np.random.default_rng(3)
    tp, dr, ds, M, P = 2, 1, 2, 4, 32
    R = tp * dr * ds
    grads = bf16(rng.normal(0, 1e-2, (M, R, P)))
    acc = oracle.reduce_bucket(tag, tp, dr, ds, P, P, grads)
    G = acc / M
    # One microbatch; replica index r' = j * dr + r; rank order keeps the
    # replica axis slowest, so the big world is the microbatches stacked.
    big = grads.reshape(1, M * R, P)
    acc_big = oracle.reduce_bucket(tag, tp, M * dr, ds, P, P, big)
    np.testing.assert_allclose(G, acc_big, rtol=1e-13, atol=1e-18)


# --------------------------------------------------------------------------
# Norm and clipping
# --------------------------------------------------------------------------
def test_norm_closed_form(orc):
    n, M, a = 1000, 4, 0.375
    acc = np.full(n, a, np.float64)
    assert oracle.norm_sq(acc, M) == n * (a / M) ** 2
    assert oracle.norm_sq(np.zeros(0), 1) == 0.0


def test_clip_special_cases(orc):
    # ||G|| <= max_norm or clipping off: coefficient exactly 1
    assert oracle.clip_coef(0.25, 1.0) == 1.0
    assert oracle.clip_coef(0.0, 1.0) == 1.0
    assert oracle.clip_coef(1e6, 0.0) == 1.0
    assert oracle.clip_coef(1e6, -1.0) == 1.0
    # above: max/(norm + 1e-6)
    assert oracle.clip_coef(4.0, 1.0) == 1.0 / (2.0 + 1e-6)
    assert math.isnan(oracle.clip_coef(float("nan"), 1.0))
    assert oracle.clip_coef(float("inf"), 1.0) == 0.0


@pytest.mark.parametrize("max_norm", [0.5, 1.0, 3.0, 100.0])
def test_clip_matches_torch_clip_grad_norm(orc, max_norm):
    rng = np.random.default_rng(4)
    arrs = [rng.normal(0, 0.3, n) for n in (17, 64, 5)]
    ts = [torch.nn.Parameter(torch.zeros(a.size, dtype=torch.float64)) for a in arrs]
    for t, a in zip(ts, arrs):
        t.grad = torch.tensor(a, dtype=torch.float64)
    total = torch.nn.utils.clip_grad_norm_(ts, max_norm, foreach=False)
    acc = np.concatenate(arrs)
    s = oracle.norm_sq(acc, 1)
    assert math.isclose(math.sqrt(s), float(total), rel_tol=1e-14)
    c = oracle.clip_coef(s, max_norm)
    clipped = np.concatenate([t.grad.numpy() for t in ts])
    np.testing.assert_allclose(c * acc, clipped, rtol=1e-14, atol=0)


# --------------------------------------------------------------------------
# AdamW
# --------------------------------------------------------------------------
HP = (1e-3, 0.9, 0.999, 1e-8, 0.01)


def test_adamw_step1_closed_form(orc):
    rng = np.random.default_rng(5)
    n = 256
    g = rng.normal(0, 1e-3, n)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    z = np.zeros(n, np.float32)
    lr, b1, b2, eps, wd = HP
    p1, m1, v1, bits = oracle.adamw(g, n, 1, 1.0, HP, 1, p0, z, z)
    want = p0.astype(np.float64) * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
    np.testing.assert_allclose(p1, want, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(m1, (1 - b1) * g, rtol=1e-6)
    np.testing.assert_allclose(v1, (1 - b2) * g * g, rtol=1e-6)


def test_adamw_zero_gradient(orc):
    rng = np.random.default_rng(6)
    n = 64
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    z = np.zeros(n, np.float32)
    p1, m1, v1, _ = oracle.adamw(np.zeros(n), n, 1, 1.0, HP, 1, p0, z, z)
    assert np.all(m1 == 0) and np.all(v1 == 0)
    np.testing.assert_array_equal(p1, (p0.astype(np.float64) * (1 - HP[0] * HP[4])).astype(np.float32))


def test_adamw_padding_written_zero(orc):
    n, used = 16, 5
    p0 = np.full(n, 0.5, np.float32)
    mv = np.full(n, 0.25, np.float32)
    p1, m1, v1, bits = oracle.adamw(np.ones(n), used, 1, 1.0, HP, 3, p0, mv, mv)
    assert np.all(p1[used:] == 0) and np.all(m1[used:] == 0) and np.all(v1[used:] == 0)
    assert np.all(bits[used:] == 0)
    assert np.all(p1[:used] != 0)


@pytest.mark.parametrize("hp", [(1e-3, 0.9, 0.999, 1e-8, 0.01), (3e-4, 0.8, 0.95, 1e-6, 0.1)])
def test_adamw_multistep_matches_torch(orc, hp):
    """Steps 1..5 against torch.optim.AdamW (fp64 CPU), with the clipped,
    microbatch-averaged gradient g = c * acc / M."""
    rng = np.random.default_rng(8)
    n, M, c = 100, 4, 0.625
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    param = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([param], lr=hp[0], betas=(hp[1], hp[2]), eps=hp[3],
                            weight_decay=hp[4], foreach=False)
    master, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for step in range(1, 6):
        acc = rng.normal(0, 1e-3, n) * M
        param.grad = torch.tensor(c * acc / M, dtype=torch.float64)
        opt.step()
        master, m, v, bits = oracle.adamw(acc, n, M, c, hp, step, master, m, v)
        ref = param.detach().numpy()
        np.testing.assert_allclose(master, ref, rtol=1e-6, atol=1e-9)
        st = opt.state[param]
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-5, atol=1e-12)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-5, atol=1e-15)
        # bf16 output is the rounded fp32 master
        np.testing.assert_array_equal(bits, bf16(master))


# --------------------------------------------------------------------------
# bf16 rounding against torch's cast
# --------------------------------------------------------------------------
def test_bf16_rne_matches_torch(orc):
    rng = np.random.default_rng(9)
    vals = np.concatenate([
        rng.normal(0, 1, 2000).astype(np.float32),
        rng.normal(0, 1e-30, 200).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38, 1e-45, 1.0 + 2 ** -8,
                  1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9], np.float32),
    ])
    # exact ties: low 16 bits = 0x8000
    ties = (rng.integers(0, 2 ** 31, 200, dtype=np.uint32) & 0xFFFF0000 | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    vals = np.concatenate([vals, ties])
    want = bf16(vals)
    got = np.array([oracle.bf16_rne(float(x)) for x in vals], np.uint16)
    np.testing.assert_array_equal(got, want)
    assert (oracle.bf16_rne(float("nan")) & 0x7FC0) == 0x7FC0


# --------------------------------------------------------------------------
# Plan: hand-derived layouts and rejections (golden/plan_layouts.json)
# --------------------------------------------------------------------------
PLAN_CASES = load("plan_layouts.json")


@pytest.mark.parametrize("case", PLAN_CASES["cases"], ids=lambda c: c["name"])
def test_plan_hand_derived(orc, case):
    p = oracle.plan(case["numel"], case["owner"], case["world"], case["tp"], case["dp_replicate"],
                    case["dp_shard"], case["bucket_bytes"], case.get("tensor_flags"))
    assert p.dp_shard == case["dp_shard_resolved"]
    for key in ("t_bucket", "t_offset", "b_tag", "b_used", "b_padded", "b_rank_off", "b_state_off"):
        assert list(getattr(p, key)) == case[key], key
    assert p.n_rank_pad == case["n_rank_pad"]
    assert p.n_state_pad == case["n_state_pad"]
    for b in range(p.n_buckets):
        assert int(p.b_padded[b]) % (8 * p.dp_shard) == 0


@pytest.mark.parametrize("case", PLAN_CASES["rejections"], ids=lambda c: c["why"])
def test_plan_rejections(orc, case):
    with pytest.raises(oracle.OracleError) as ei:
        oracle.plan(case["numel"], case["owner"], case["world"], case["tp"], case["dp_replicate"],
                    case["dp_shard"], case["bucket_bytes"], case.get("tensor_flags"))
    assert ei.value.code == case["status"]


def test_plan_workload_invariants(orc):
    """Each tensor sits in exactly one bucket of its own tag, without
    overlap; LOCAL_SHARD takes numel/tp per rank; buckets respect the byte
    cap unless they hold a single tensor."""
    import workloads
    for cid in workloads.ALL_IDS:
        w = workloads.get(cid)
        p = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard,
                        w.bucket_bytes)
        members = {b: [] for b in range(p.n_buckets)}
        for i, t in enumerate(w.tensors):
            b = int(p.t_bucket[i])
            assert int(p.b_tag[b]) == t.owner
            per_rank = t.numel // w.tp if t.owner == LOCAL_SHARD else t.numel
            members[b].append((int(p.t_offset[i]), per_rank))
        for b, segs in members.items():
            segs.sort()
            pos = 0
            for off, n in segs:
                assert off == pos
                pos += n
            assert pos == int(p.b_used[b])
            if len(segs) > 1:
                assert 2 * pos <= w.bucket_bytes
        n_unique = sum(int(p.b_used[b]) * p.copies(b) for b in range(p.n_buckets))
        assert n_unique == w.n_unique


# --------------------------------------------------------------------------
# Unused parameters (grad None) and frozen parameters against torch
# --------------------------------------------------------------------------
def test_masked_update_matches_torch_grad_none_semantics(orc):
    """Four steps on a world-1 plan (the reduction is the identity), some
    tensors without a gradient in some steps, one frozen tensor: the oracle's
    masked update equals clip_grad_norm_ + torch.optim.AdamW, which skip
    parameters whose grad is None (norm, moments, weight decay, step)."""
    rng = np.random.default_rng(21)
    numels = [24, 7, 16, 5]
    flags = [0, 0, oracle_frozen(), 0]
    hp = (1e-2, 0.9, 0.99, 1e-8, 0.05)
    max_norm = 0.05
    p = oracle.plan(numels, [REPLICA_AVG] * 4, 1, 1, 1, 1, 1 << 20, flags)
    p0 = [rng.normal(0, 0.02, n).astype(np.float32) for n in numels]
    params = [torch.nn.Parameter(torch.tensor(x, dtype=torch.float64)) for x in p0]
    params[2].requires_grad_(False)
    trainable = [params[i] for i in (0, 1, 3)]
    opt = torch.optim.AdamW(trainable, lr=hp[0], betas=(hp[1], hp[2]), eps=hp[3], weight_decay=hp[4],
                            foreach=False)
    nsp = p.n_state_pad
    master = np.zeros(nsp, np.float32)
    for i in range(4):
        for lo, hi in p.tensor_rows(i):
            master[lo:hi] = p0[i]
    m = np.zeros(nsp, np.float32)
    v = np.zeros(nsp, np.float32)
    bits = np.zeros(nsp, np.uint16)
    steps = [0, 0, 0, 0]
    masks = [[1, 1, 0, 1], [1, 0, 0, 1], [0, 1, 0, 1], [1, 1, 0, 0]]
    for used in masks:
        grads = [rng.normal(0, 0.03, n).astype(np.float32) for n in numels]
        for i, prm in enumerate(params):
            if i == 2:
                continue
            prm.grad = torch.tensor(grads[i], dtype=torch.float64) if used[i] else None
        torch.nn.utils.clip_grad_norm_(trainable, max_norm, foreach=False)
        opt.step()
        host = np.zeros(p.n_rank_pad, np.float32)
        for i in range(4):
            b = int(p.t_bucket[i])
            if b >= 0:
                o = int(p.b_rank_off[b]) + int(p.t_offset[i])
                host[o:o + numels[i]] = grads[i]

        def grads_of(b, host=host):
            ro, P = int(p.b_rank_off[b]), int(p.b_padded[b])
            return host[ro:ro + P].reshape(1, 1, P)

        res, steps = oracle.full_update_masked(p, grads_of, 1, hp, max_norm, used, steps, master, m, v, bits)
        master, m, v, bits = res.master, res.m, res.v, res.params_bf16
        for i in (0, 1, 3):
            (lo, hi), = p.tensor_rows(i)
            np.testing.assert_allclose(master[lo:hi], params[i].detach().numpy(), rtol=1e-6, atol=1e-9)
            st = opt.state[params[i]]
            if st:
                # the oracle stores fp32 moments between steps; near a cancellation
                # that rounding is absolute (~1e-10 for moments of size 1e-3)
                np.testing.assert_allclose(m[lo:hi], st["exp_avg"].numpy(), rtol=1e-5, atol=1e-9)
                np.testing.assert_allclose(v[lo:hi], st["exp_avg_sq"].numpy(), rtol=1e-5, atol=1e-13)
                assert steps[i] == int(st["step"])
        assert p.tensor_rows(2) == []
    assert np.array_equal(params[2].detach().numpy(), p0[2].astype(np.float64))


def oracle_frozen():
    return 1


def test_logical_layout_hand_derived(orc):
    """The odd-size tiny plan (golden 'odd-sizes-ds2'): state = its own index.
    Logical order: tensor 0 (RA, 21) = state[0:21]; tensor 1 (PS, 5) =
    state[32:37]; tensor 2 (LS, 18: 9 per tp row) = rows t=0 state[48:57]
    then t=1 state[64:73]; tensor 3 (AR, 3) = state[80:83]."""
    p = oracle.plan([21, 5, 18, 3], [0, 1, 2, 3], 4, 2, 1, 2, 26214400)
    st = np.arange(p.n_state_pad, dtype=np.float32)
    want = np.concatenate([np.arange(0, 21), np.arange(32, 37), np.arange(48, 57), np.arange(64, 73),
                           np.arange(80, 83)]).astype(np.float32)
    lg = oracle.to_logical(p, st)
    assert np.array_equal(lg, want)
    back = oracle.from_logical(p, lg)
    keep = np.zeros(p.n_state_pad, bool)
    keep[want.astype(int)] = True
    assert np.array_equal(back[keep], st[keep]) and np.all(back[~keep] == 0)


def test_gather_tensor_bf16_hand_derived(orc):
    """oracle.gather_tensor (bf16 parameters) on a hand-laid-out plan whose
    buckets hold two tensors of the same tag, so tensors sit at nonzero
    offsets inside their bucket.  Plan [21 RA, 5 PS, 18 LS, 3 AR, 10 LS,
    7 RA], tp 2, dp_shard 2, one bucket per tag (padding quantum 8 * 2):
      RA bucket: tensor 0 at 0 (21), tensor 5 at 21 (7); used 28, padded 32;
                 state [0, 32)
      PS bucket: tensor 1 at 0 (5); padded 16; state [32, 48)
      LS bucket: per tp row tensor 2 at 0 (9), tensor 4 at 9 (5); used 14,
                 padded 16; rows t = 0, 1 at state 48 and 64
      AR bucket: tensor 3 at 0 (3); padded 16; state [80, 96)
    With every parameter equal to its own state index, the gathered tensors
    are those indices: a LOCAL_SHARD tensor is row 0's chunk then row 1's
    (its dim-0 halves) at state_off + t * padded + offset ("Cosmos 3 ...
    distributed parallelism", section 2: all-gather of the shards)."""
    p = oracle.plan([21, 5, 18, 3, 10, 7], [REPLICA_AVG, PARTIAL_SUM, LOCAL_SHARD, ALREADY_REDUCED,
                                            LOCAL_SHARD, REPLICA_AVG], 4, 2, 1, 2, 25 << 20)
    assert list(p.b_state_off) == [0, 32, 48, 80] and list(p.b_padded) == [32, 16, 16, 16]
    assert list(p.t_offset) == [0, 0, 0, 0, 9, 21] and p.n_state_pad == 96
    params = np.arange(p.n_state_pad, dtype=np.uint16)
    want = {0: np.arange(0, 21), 1: np.arange(32, 37), 2: np.r_[48:57, 64:73], 3: np.arange(80, 83),
            4: np.r_[57:62, 73:78], 5: np.arange(21, 28)}
    for i, w in want.items():
        got = oracle.gather_tensor(p, i, params)
        assert got.dtype == np.uint16 and np.array_equal(got, w.astype(np.uint16)), (i, got, w)
    # the fp32 twin places every tensor in the same way
    st = np.arange(p.n_state_pad, dtype=np.float32)
    assert np.array_equal(oracle.to_logical(p, st),
                          np.concatenate([want[i] for i in range(6)]).astype(np.float32))


# --------------------------------------------------------------------------
# The fp32 accumulation error bound that widens the master/moment checks
# (oracle.accumulation_error_bound).  Each case evaluates the accumulator
# the way an fp32 implementation may (per microbatch the group's bf16 values
# summed left to right in fp32, times the fp32 scale, added into an fp32
# accumulator), computes the exact value in rational arithmetic, and checks
# the error against the bound the oracle gives from the absolute inputs.
# --------------------------------------------------------------------------
TINY = 2.0 ** -25 * (1 + 2.0 ** -7)  # bf16, under half an fp32 ulp of 1.0 (TINY / 2: of 0.5)


def _fp32_eval(vals, scale):
    """vals [M][group] (floats exactly representable in bf16) -> fp32 acc."""
    sc = np.float32(scale)
    acc = np.float32(0.0)
    for j, row in enumerate(vals):
        s = np.float32(row[0])
        for x in row[1:]:
            s = np.float32(s + np.float32(x))
        p_ = np.float32(s * sc)
        acc = p_ if j == 0 else np.float32(acc + p_)
    return float(acc)


def _exact(vals, group):
    from fractions import Fraction
    return Fraction(sum(Fraction(float(x)) for row in vals for x in row)) / group


def _bound_case(vals):
    """(|fp32 - exact|, delta) for one REPLICA_AVG element over a world of
    `group` ranks (tp 1, dp_replicate = group, dp_shard 1: scale 1/group)."""
    vals = np.asarray(vals, np.float64)
    M, R = vals.shape
    bits = bf16(vals.reshape(M, R, 1))
    assert np.array_equal(bits_to_f32(bits).astype(np.float64).reshape(M, R), vals), "not bf16"
    g = np.zeros((M, R, 8), np.uint16)
    g[:, :, 0] = bits[:, :, 0]
    acc = oracle.reduce_bucket(REPLICA_AVG, 1, R, 1, 8, 1, g)
    ab = oracle.reduce_bucket(REPLICA_AVG, 1, R, 1, 8, 1, oracle.abs_inputs(g))
    delta = float(oracle.accumulation_error_bound(ab, M, R)[0, 0])
    exact = _exact(vals, R)
    assert abs(acc[0, 0] - float(exact)) <= 1e-15 * float(ab[0, 0])  # the fp64 oracle itself
    return abs(_fp32_eval(vals, 1.0 / R) - float(exact)), delta


def test_accumulation_bound_absorption_across_ranks(orc):
    """1.0 on rank 0 and TINY on each of the 15 others: every fp32 addition
    rounds TINY away, an error of 15 TINY = 7.6 u of the sum of |terms|.
    The bound must cover it (a bound without the group's additions, e.g.
    (M + 2) u, would not) and not exceed it by more than 3x."""
    err, delta = _bound_case([[1.0] + [TINY] * 15])
    assert 0 < err <= delta
    assert err >= delta / 3
    assert err > 3 * 2.0 ** -24 * (1 + 15 * TINY) / 16  # what (M + 2) u would allow


def test_accumulation_bound_absorption_across_microbatches(orc):
    """Two ranks, 16 microbatches: the first brings 0.5 into the
    accumulator, each later one TINY / 2, which rounds away: the error grows
    with M, and the bound must grow with it (a bound without M would not
    cover it)."""
    vals = [[1.0, 0.0]] + [[TINY, 0.0]] * 15
    err, delta = _bound_case(vals)
    assert 0 < err <= delta
    assert err >= delta / 3
    assert err > oracle.gamma(2 + 1) * (1 + 15 * TINY) / 2  # a bound without the M term


def test_accumulation_bound_uses_absolute_values(orc):
    """1 + TINY - 1: the fp32 sum is 0, the exact one TINY / 3.  The signed
    sum of the terms is TINY / 3, far too small to bound the error: the bound
    must be taken from the absolute values."""
    err, delta = _bound_case([[1.0, TINY, -1.0]])
    assert err == TINY / 3
    assert err <= delta
    assert err > oracle.gamma(3 + 1 + 1) * (TINY / 3)


@pytest.mark.parametrize("R,M", [(16, 1), (12, 3), (4, 8), (128, 1)])
def test_accumulation_bound_random_cancelling(orc, R, M):
    """Random bf16 values with exponents spread over 2^-24..1 and adjacent
    ranks nearly cancelling (x, -x (1 - 2^-8)): every fp32 evaluation stays
    within the bound."""
    rng = np.random.default_rng(R * 100 + M)
    worst = 0.0
    for _ in range(300):
        mag = 2.0 ** rng.integers(-24, 1, (M, R)) * (1 + rng.integers(0, 128, (M, R)) / 128)
        sign = rng.choice([-1.0, 1.0], (M, R))
        vals = mag * sign
        vals[:, 1::2] = -vals[:, 0:R - R % 2:2] * (1 - 2.0 ** -8)
        vals = bits_to_f32(bf16(vals)).astype(np.float64)
        err, delta = _bound_case(vals)
        assert err <= delta, (vals, err, delta)
        worst = max(worst, err / delta)
    assert worst < 1.0


def test_gamma_closed_form(orc):
    """gamma_k = k u / (1 - k u) with u = 2^-24."""
    u = 2.0 ** -24
    for k in (1, 3, 18, 133):
        assert oracle.gamma(k) == k * u / (1 - k * u)
    assert oracle.gamma(0) == 0.0
