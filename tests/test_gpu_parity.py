"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs, element by element, at sizes the oracle finishes in
seconds that still span many tiles and ragged tails.

Tolerances (fp32 accumulator/norm/master/moments rel 1e-5 + abs 1e-7, bf16
parameters within 1 ulp; routing, offsets and padding bit-exact).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_support import (Case, Run, assert_bf16_cast, assert_close, assert_close_bracketed,
                         assert_within_accumulation_bound, case_from_workload, grs, oracle_update,
                         padding_mask)

pytestmark = pytest.mark.gpu

RA, PS, LS, AR = 0, 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.init()


def full_check(run: Run, res, what="", acc_where=None):
    """Everything the update wrote against the oracle; `acc_where` (bool per
    state element) limits the accumulator check (a masked reduction leaves
    the accumulator of tensors without a gradient unspecified)."""
    torch.cuda.synchronize()
    n = run.nsp
    pad = padding_mask(run.op)
    acc = run.acc[:n].cpu().numpy()
    if acc_where is None:
        assert_close(acc, res.acc, f"{what} acc")
    else:
        assert_close(acc[acc_where], res.acc[acc_where], f"{what} acc")
    if res.delta is not None:  # the bound behind the master/moment brackets holds on the kernel
        w = np.ones(n, bool) if acc_where is None else acc_where
        assert_within_accumulation_bound(acc[w], res.acc[w], res.delta[w], f"{what} acc")
    assert np.all(acc[pad] == 0), f"{what} acc padding not zero"
    norm = float(run.norm.cpu()[0])
    assert_close([norm], [res.norm_sq], f"{what} norm_sq")
    master, m, v = run.state_host()
    if res.lo is not None:
        for name, got, want, lo, hi in zip(("master", "m", "v"), (master, m, v), (res.master, res.m, res.v),
                                           res.lo, res.hi):
            assert_close_bracketed(got, want, lo, hi, f"{what} {name}")
    else:
        assert_close(master, res.master, f"{what} master")
        assert_close(m, res.m, f"{what} m")
        assert_close(v, res.v, f"{what} v")
    for name, arr in (("master", master), ("m", m), ("v", v)):
        assert np.all(arr[pad] == 0), f"{what} {name} padding not zero"
    bits = run.params[:n].cpu().numpy().view(np.uint16)
    lo_p, hi_p = (res.lo[0], res.hi[0]) if res.lo is not None else (None, None)
    assert_bf16_cast(bits, master, res.params_bf16, res.master, f"{what} params", lo_master=lo_p, hi_master=hi_p)
    assert np.all(bits[pad] == 0)


def small_cases():
    cases = {"tiny-world4": case_from_workload(0)}
    base = dict(world=4, tp=2, dp_replicate=1, dp_shard=2, bucket_bytes=25 << 20)
    cases["odd-ds2"] = Case([21, 5, 18, 3], [RA, PS, LS, AR], n_micro=1, grad_std=1e-2,
                            seed_base=11, **base)
    cases["odd-ds3-M3"] = Case([21, 5, 18, 3, 1001, 77], [RA, PS, LS, AR, RA, PS], 6, 2, 1, 3,
                               256, 3, 1e-2, 12)
    # many tiles + ragged tails: buckets of 10^5.. elements, R up to 16
    cases["multi-tile-world16-M2"] = Case(
        [100003, 1024, 65536 * 2, 4099, 333, 70001, 8 * 1000], [RA, PS, LS, AR, PS, RA, LS],
        16, 2, 2, 4, 1 << 18, 2, 1e-3, 13)
    cases["tp4-world8"] = Case([40000, 4096 * 4, 2000, 12], [RA, LS, PS, AR], 8, 4, 1, 2, 1 << 16,
                               1, 1e-3, 14)
    cases["world1"] = Case([5000, 17, 300], [RA, PS, AR], 1, 1, 1, 1, 4096, 2, 1e-2, 15)
    cases["world3-non-pow2"] = Case([3001, 99, 330], [RA, PS, LS], 3, 1, 3, 1, 2048, 3, 1e-3, 16)
    cases["world6-auto-shard"] = Case([5000, 600, 36], [RA, LS, PS], 6, 2, 1, -1, 8192, 1, 1e-3, 17)
    # fp32 gradient input (plan flag), many tiles, ragged tails, 3 microbatches
    cases["fp32-grads-world8-M3"] = Case(
        [70001, 1000, 40000 * 2, 77, 9999], [RA, PS, LS, AR, RA], 8, 2, 2, 2, 1 << 17, 3, 1e-3, 18,
        fp32_grads=True)
    # maximum world (128 ranks: 1 KB-per-rank tiles) and 64 ranks with tp 4
    cases["world128-max"] = Case([30001, 512, 4096 * 2, 100], [RA, PS, LS, AR], 128, 2, 8, 8, 1 << 16, 1,
                                 1e-3, 22)
    cases["world64-tp4-M2"] = Case([20000, 300, 4096 * 4, 9], [RA, PS, LS, AR], 64, 4, 4, 4, 1 << 15, 2,
                                   1e-3, 23)
    # degenerate: zero-size tensors, a bucket holding only zero-size tensors (no tiles)
    cases["zero-size-tensors"] = Case([0, 1000, 0, 64, 0], [RA, RA, PS, AR, LS], 2, 1, 1, 2, 1 << 20, 1,
                                      1e-2, 24)
    # many small tensors of all four tags (3000, 1..400 elements): most tiles
    # span several tensors, the gather needs several launches (256 pointers each)
    rng = np.random.default_rng(2024)
    owners_many = rng.integers(0, 4, 3000).tolist()
    numels_many = [int(x) * (2 if o == LS else 1) for x, o in zip(rng.integers(1, 201, 3000), owners_many)]
    cases["many-small-tensors"] = Case(numels_many, owners_many, 8, 2, 2, 2, 1 << 16, 1, 1e-2, 25)
    cases["fp32-grads-world16"] = Case(
        [100003, 1024, 65536 * 2, 4099], [RA, PS, LS, AR], 16, 2, 2, 4, 1 << 18, 1, 1e-3, 19,
        fp32_grads=True)
    return cases


SMALL = small_cases()


@pytest.mark.parametrize("name", list(SMALL))
def test_update_matches_oracle(name):
    c = SMALL[name]
    run = Run(c)
    try:
        master0, m0, v0 = run.state_host()
        run.update()
        assert run.check_flags() == 0
        res = oracle_update(run, master0, m0, v0, step=1)
        full_check(run, res, name)
    finally:
        run.close()


@pytest.mark.parametrize("name", ["tiny-world4", "multi-tile-world16-M2"])
def test_three_steps_match_oracle(name):
    """Step counting, bias correction and carried moments (new grads each step)."""
    c = SMALL[name]
    run = Run(c)
    try:
        master, m, v = run.state_host()  # initial state: seeded inputs
        for step in range(1, 4):
            if step > 1:
                run.fill_grads(step_seed=step)
            run.update()
            res = oracle_update(run, master, m, v, step=step)
            full_check(run, res, f"{name} step {step}")
            master, m, v = res.master, res.m, res.v  # the oracle carries its own state
    finally:
        run.close()


def test_forty_steps_track_the_oracle():
    """Forty updates with new gradients each step, the oracle carrying its
    own fp64-evaluated state rounded to fp32 after every step: step counting
    and bias correction stay right as the corrections decay, and the fp32
    evaluation does not drift from the fp64 one beyond the tolerance."""
    c = SMALL["odd-ds3-M3"]
    run = Run(c)
    try:
        master, m, v = run.state_host()
        for step in range(1, 41):
            if step > 1:
                run.fill_grads(step_seed=step)
            run.update()
            res = oracle_update(run, master, m, v, step=step)
            if step % 10 == 0 or step < 3:
                full_check(run, res, f"step {step}")
            master, m, v = res.master, res.m, res.v
    finally:
        run.close()


@pytest.mark.parametrize("name", ["odd-ds3-M3", "multi-tile-world16-M2"])
def test_clip_off_matches_oracle(name):
    c = SMALL[name]
    run = Run(c)
    try:
        master0, m0, v0 = run.state_host()
        run.update(max_norm=0.0)
        res = oracle_update(run, master0, m0, v0, step=1, max_norm=0.0)
        full_check(run, res, name + " clip off")
    finally:
        run.close()


def test_per_bucket_equals_grouped_and_fused_norm_equals_pass1():
    """grs_reduce_bucket == grs_reduce_all bit for bit; the fused norm
    partials == the separate pass over acc bit for bit; reruns identical."""
    c = SMALL["multi-tile-world16-M2"]
    run = Run(c)
    try:
        run.reduce(per_bucket=False)
        run.norm_sq(partials_ready=True)
        torch.cuda.synchronize()
        acc_a = run.acc.clone()
        norm_a = run.norm.clone()
        run.acc.fill_(123.0)
        run.reduce(per_bucket=True)
        run.norm_sq(partials_ready=True)
        torch.cuda.synchronize()
        assert torch.equal(acc_a, run.acc)
        assert torch.equal(norm_a, run.norm)
        run.norm.zero_()
        run.norm_sq(partials_ready=False)
        torch.cuda.synchronize()
        assert torch.equal(norm_a, run.norm)
        # determinism of the whole update
        outs = []
        for _ in range(2):
            run2 = Run(c)
            try:
                run2.update()
                torch.cuda.synchronize()
                outs.append([t.clone() for t in (run2.acc, run2.norm, run2.master, run2.m, run2.v,
                                                 run2.params)])
            finally:
                run2.close()
        for a, b in zip(*outs):
            assert torch.equal(a, b)
    finally:
        run.close()


def test_owner_routing_is_exact():
    """Routing pins on the GPU: identical rank copies give exact RA/LS/AR
    values and tp x the value for PS; perturbing non-canonical ranks of an
    ALREADY_REDUCED bucket or another tp index of a LOCAL_SHARD bucket
    leaves those outputs bit-identical."""
    c = Case([4096, 512, 2048 * 2, 96], [RA, PS, LS, AR], 8, 2, 2, 2, 1 << 20, 1, 1e-2, 21)
    run = Run(c)
    try:
        base = run.grads[0][0].clone()
        for k in range(c.world):
            run.grads[0][k].copy_(base)
        run.reduce()
        torch.cuda.synchronize()
        acc = run.acc.clone()
        x = base.float()
        for b in range(run.op.n_buckets):
            tag = int(run.op.b_tag[b])
            P = int(run.op.b_padded[b])
            ro, so, used = int(run.op.b_rank_off[b]), int(run.op.b_state_off[b]), int(run.op.b_used[b])
            want = x[ro:ro + used] * (c.tp if tag == PS else 1)
            for t in range(run.op.copies(b)):
                got = acc[so + t * P: so + t * P + used]
                assert torch.equal(got, want), (b, tag, t)
        # perturb: AR non-canonical ranks, LS ranks of tp index 1
        gen = torch.Generator(device="cuda").manual_seed(5)
        for k in range(1, c.world):
            noise = (torch.randn(run.nrp, generator=gen, device="cuda") * 0.1).to(torch.bfloat16)
            for b in range(run.op.n_buckets):
                tag = int(run.op.b_tag[b])
                ro, used = int(run.op.b_rank_off[b]), int(run.op.b_used[b])
                if tag == AR or (tag == LS and k % c.tp == 1):
                    run.grads[0][k][ro:ro + used] = noise[ro:ro + used]
        run.reduce()
        torch.cuda.synchronize()
        for b in range(run.op.n_buckets):
            tag = int(run.op.b_tag[b])
            P, so = int(run.op.b_padded[b]), int(run.op.b_state_off[b])
            if tag == AR:
                assert torch.equal(acc[so:so + P], run.acc[so:so + P])
            if tag == LS:
                assert torch.equal(acc[so:so + P], run.acc[so:so + P])          # row t=0 unchanged
                assert not torch.equal(acc[so + P:so + 2 * P], run.acc[so + P:so + 2 * P])
            if tag in (RA, PS):
                assert torch.equal(acc[so:so + P], run.acc[so:so + P])  # only AR/LS ranks perturbed
    finally:
        run.close()


def test_gather_matches_oracle():
    for name in ("tiny-world4", "odd-ds3-M3", "multi-tile-world16-M2", "many-small-tensors"):
        c = SMALL[name]
        run = Run(c)
        try:
            run.update()
            torch.cuda.synchronize()
            outs = [torch.full((max(n, 1),), -1, dtype=torch.int16, device="cuda") for n in c.numels]
            # odd offsets inside a larger buffer exercise the unaligned paths
            big = torch.full((sum(c.numels) + len(c.numels) + 64,), -1, dtype=torch.int16, device="cuda")
            ptrs, views, off = [], [], 3
            for n in c.numels:
                assert off + n <= big.numel()  # every destination inside the buffer
                views.append(big[off:off + n])
                ptrs.append(big.data_ptr() + 2 * off)
                off += n + 1
            grs().grs_gather_params(run.plan, run.params.data_ptr(), [t.data_ptr() for t in outs],
                                    run.stream())
            grs().grs_gather_params(run.plan, run.params.data_ptr(), ptrs, run.stream())
            torch.cuda.synchronize()
            params = run.params[:run.nsp].cpu().numpy().view(np.uint16)
            for i, n in enumerate(c.numels):
                want = oracle.gather_tensor(run.op, i, params)
                got = outs[i][:n].cpu().numpy().view(np.uint16)
                assert np.array_equal(got, want), (name, i)
                got2 = views[i].cpu().numpy().view(np.uint16)
                assert np.array_equal(got2, want), (name, i, "unaligned")
        finally:
            run.close()


@pytest.mark.parametrize("name", ["tiny-world4", "odd-ds3-M3", "multi-tile-world16-M2", "tp4-world8",
                                  "many-small-tensors", "zero-size-tensors", "fp32-grads-world8-M3",
                                  "world128-max", "world6-auto-shard"])
def test_update_to_tensors_matches_update_then_gather(name):
    """grs_clip_adamw_step_to_tensors (the gather fused into the update):
    (1) with the bucket-ordered buffer as well: master, m, v and that buffer
    equal grs_clip_adamw_step's bit for bit, the whole update matches the
    oracle, and every tensor equals oracle.gather_tensor of the buffer bit
    for bit, at 16-byte-aligned and at odd 2-byte offsets; (2) without the
    buffer (NULL): the same tensors, the buffer untouched; NULL table
    entries leave their tensors untouched."""
    g = grs()
    c = SMALL[name]
    ref, run, bare = Run(c), Run(c), Run(c)
    try:
        master0, m0, v0 = run.state_host()
        ref.update()
        n_t = len(c.numels)
        outs = [torch.full((max(n, 1),), -1, dtype=torch.int16, device="cuda") for n in c.numels]
        big = torch.full((sum(c.numels) + n_t + 64,), -1, dtype=torch.int16, device="cuda")
        views, odd_ptrs, off = [], [], 3
        for n in c.numels:
            assert off + n <= big.numel()  # every destination inside the buffer
            views.append(big[off:off + n])
            odd_ptrs.append(big.data_ptr() + 2 * off)
            off += n + 1
        table = torch.tensor([t.data_ptr() for t in outs], dtype=torch.int64, device="cuda")
        table_odd = torch.tensor(odd_ptrs, dtype=torch.int64, device="cuda")
        hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], c.max_norm, 1, c.n_micro)
        # (1) bucket-ordered buffer and per-tensor storage (aligned, then odd offsets)
        run.reduce()
        run.norm_sq()
        m_save, v_save, p_save = run.m.clone(), run.v.clone(), run.master.clone()
        g.grs_clip_adamw_step_to_tensors(run.plan, hp, run.norm.data_ptr(), run.acc.data_ptr(),
                                         run.master.data_ptr(), run.m.data_ptr(), run.v.data_ptr(),
                                         run.params.data_ptr(), table.data_ptr(), run.stream())
        torch.cuda.synchronize()
        for nm in ("acc", "norm", "master", "m", "v", "params"):
            assert torch.equal(getattr(ref, nm), getattr(run, nm)), nm
        run.step = 1
        full_check(run, oracle_update(run, master0, m0, v0, step=1), f"{name} to tensors")
        params = run.params[:run.nsp].cpu().numpy().view(np.uint16)
        want = [oracle.gather_tensor(run.op, i, params) for i in range(n_t)]
        for i, n in enumerate(c.numels):
            assert np.array_equal(outs[i][:n].cpu().numpy().view(np.uint16), want[i]), (name, i)
        # the same update again from the saved state, into the odd offsets
        run.master.copy_(p_save)
        run.m.copy_(m_save)
        run.v.copy_(v_save)
        g.grs_clip_adamw_step_to_tensors(run.plan, hp, run.norm.data_ptr(), run.acc.data_ptr(),
                                         run.master.data_ptr(), run.m.data_ptr(), run.v.data_ptr(),
                                         run.params.data_ptr(), table_odd.data_ptr(), run.stream())
        torch.cuda.synchronize()
        assert torch.equal(ref.master, run.master) and torch.equal(ref.params, run.params)
        for i, n in enumerate(c.numels):
            assert np.array_equal(views[i].cpu().numpy().view(np.uint16), want[i]), (name, i, "odd")
        outside = torch.ones(big.numel(), dtype=torch.bool, device="cuda")
        off = 3
        for n in c.numels:
            outside[off:off + n] = False
            off += n + 1
        assert bool((big[outside] == -1).all()), (name, "write between or around the tensors")
        # (2) per-tensor storage only; every other table entry NULL
        bare.reduce()
        bare.norm_sq()
        bare.params.fill_(-7)
        outs2 = [torch.full((max(n, 1),), -1, dtype=torch.int16, device="cuda") for n in c.numels]
        table2 = torch.tensor([t.data_ptr() if i % 2 == 0 else 0 for i, t in enumerate(outs2)],
                              dtype=torch.int64, device="cuda")
        g.grs_clip_adamw_step_to_tensors(bare.plan, hp, bare.norm.data_ptr(), bare.acc.data_ptr(),
                                         bare.master.data_ptr(), bare.m.data_ptr(), bare.v.data_ptr(),
                                         None, table2.data_ptr(), bare.stream())
        torch.cuda.synchronize()
        assert bare.check_flags() == 0
        assert torch.equal(ref.master, bare.master) and torch.equal(ref.v, bare.v)
        assert bool((bare.params == -7).all())
        for i, n in enumerate(c.numels):
            got = outs2[i][:n].cpu().numpy().view(np.uint16)
            if i % 2 == 0:
                assert np.array_equal(got, want[i]), (name, i, "no bucket buffer")
            else:
                assert np.all(got == 0xFFFF), (name, i, "NULL entry written")
    finally:
        ref.close()
        run.close()
        bare.close()


def test_update_to_tensors_argument_errors():
    g = grs()
    run = Run(SMALL["odd-ds2"])
    try:
        c = run.c
        hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], c.max_norm, 1, c.n_micro)
        table = torch.zeros(len(c.numels) + 1, dtype=torch.int64, device="cuda")
        args = [run.plan, hp, run.norm.data_ptr(), run.acc.data_ptr(), run.master.data_ptr(),
                run.m.data_ptr(), run.v.data_ptr(), run.params.data_ptr(), table.data_ptr(), run.stream()]
        for k, bad, status in ((8, 0, g.GRS_ERR_INVALID_ARG), (8, table.data_ptr() + 4, g.GRS_ERR_ALIGNMENT),
                               (7, run.params.data_ptr() + 2, g.GRS_ERR_ALIGNMENT),
                               (3, run.acc.data_ptr() + 4, g.GRS_ERR_ALIGNMENT)):
            a = list(args)
            a[k] = bad
            with pytest.raises(g.GrsError) as ei:
                g.grs_clip_adamw_step_to_tensors(*a)
            assert ei.value.status == status, (k, ei.value)
        hp0 = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], c.max_norm, 0, c.n_micro)
        with pytest.raises(g.GrsError) as ei:
            g.grs_clip_adamw_step_to_tensors(run.plan, hp0, *args[2:])
        assert ei.value.status == g.GRS_ERR_INVALID_ARG
    finally:
        run.close()


def check_shard_views(run, c, master0, m0, v0, label):
    """Each rank's shard view (grs_plan_shard_view) given that rank's slices
    of the plan's reduced gradient and of the state before the update
    (device tensors master0, m0, v0; `run` has taken its one update): the
    squared norms of the views of one replica add up to the plan's S (the
    one scalar all-reduce), and clip + AdamW + bf16 on each view with that S
    equals the plan's own update restricted to the rank's elements, bit for
    bit -- so an all-gather of the views' bf16 shards gives the plan's
    parameters ("Cosmos 3 ... distributed parallelism", section 2).  A view
    refuses the reductions."""
    g = grs()
    full = {k: getattr(run, k)[:run.nsp] for k in ("acc", "master", "m", "v", "params")}
    info = run.info
    bks = [g.grs_bucket_info(run.plan, b) for b in range(info["n_buckets"])]
    s_sum = 0.0
    hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], c.max_norm, 1, c.n_micro)
    for t in range(c.tp):
        for s in range(info["dp_shard"]):
            view = g.grs_plan_shard_view(run.plan, s, t)
            try:
                vi = g.grs_plan_query(view)
                idx = []
                for pb in bks:
                    row = t if pb["tag"] == LS else 0
                    L = int(pb["shard_len"])
                    base = int(pb["state_offset"]) + row * int(pb["padded"]) + s * L
                    idx.append(torch.arange(base, base + L, device="cuda"))
                idx = torch.cat(idx) if idx else torch.zeros(0, dtype=torch.int64, device="cuda")
                assert idx.numel() == vi["n_state_pad"]
                n = max(8, idx.numel())
                acc_v = torch.zeros(n, device="cuda")
                acc_v[:idx.numel()] = full["acc"][idx]
                st = [torch.zeros(n, device="cuda") for _ in range(3)]
                for x, src in zip(st, (master0, m0, v0)):
                    x[:idx.numel()] = src[idx]
                params_v = torch.full((n,), -1, dtype=torch.int16, device="cuda")
                ws = torch.zeros(max(vi["workspace_bytes"], 16) // 4 + 4, device="cuda")
                nv = torch.zeros(1, dtype=torch.float64, device="cuda")
                g.grs_grad_norm_sq(view, acc_v.data_ptr(), c.n_micro, ws.data_ptr(), 0, nv.data_ptr(), run.stream())
                g.grs_clip_adamw_step(view, hp, run.norm.data_ptr(), acc_v.data_ptr(), st[0].data_ptr(),
                                      st[1].data_ptr(), st[2].data_ptr(), params_v.data_ptr(), run.stream())
                torch.cuda.synchronize()
                assert g.grs_check_device_errors(view, run.stream()) == 0
                k = idx.numel()
                for x, nm in zip(st, ("master", "m", "v")):
                    assert torch.equal(x[:k], full[nm][idx]), (label, s, t, nm)
                assert torch.equal(params_v[:k], full["params"][idx]), (label, s, t, "params")
                s_sum += float(nv.cpu()[0])
                with pytest.raises(g.GrsError) as ei:
                    g.grs_reduce_all(view, run.ptrs(0), acc_v.data_ptr(), 0, 0, ws.data_ptr(), run.stream())
                assert ei.value.status == g.GRS_ERR_UNSUPPORTED_COMPOSITION
                with pytest.raises(g.GrsError) as ei:
                    g.grs_grad_norm_sq(view, acc_v.data_ptr(), c.n_micro, ws.data_ptr(), 1, nv.data_ptr(),
                                       run.stream())
                assert ei.value.status == g.GRS_ERR_UNSUPPORTED_COMPOSITION
            finally:
                g.grs_plan_destroy(view)
    want = float(run.norm.cpu()[0])
    assert abs(s_sum - want) <= 1e-5 * want, (label, s_sum, want)


def check_update_to_tensors(c, label):
    """grs_clip_adamw_step_to_tensors with per-tensor storage only (no
    bucket-ordered buffer) after the plain reduction and norm: master, m and
    v equal grs_clip_adamw_step's bit for bit, every tensor equals
    oracle.gather_tensor of that update's bucket-ordered buffer bit for bit,
    and frozen tensors (not in the plan) are left untouched."""
    g = grs()
    ref, run = Run(c), Run(c)
    try:
        ref.update()
        run.reduce()
        run.norm_sq()
        outs = [torch.full((max(n, 1),), -1, dtype=torch.int16, device="cuda") for n in c.numels]
        table = torch.tensor([t.data_ptr() for t in outs], dtype=torch.int64, device="cuda")
        hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], c.max_norm, 1, c.n_micro)
        g.grs_clip_adamw_step_to_tensors(run.plan, hp, run.norm.data_ptr(), run.acc.data_ptr(),
                                         run.master.data_ptr(), run.m.data_ptr(), run.v.data_ptr(),
                                         None, table.data_ptr(), run.stream())
        torch.cuda.synchronize()
        assert run.check_flags() == 0
        for nm in ("master", "m", "v"):
            assert torch.equal(getattr(ref, nm)[:ref.nsp], getattr(run, nm)[:run.nsp]), (label, nm)
        params = ref.params[:ref.nsp].cpu().numpy().view(np.uint16)
        for i, n in enumerate(c.numels):
            got = outs[i][:n].cpu().numpy().view(np.uint16)
            if int(ref.op.t_bucket[i]) < 0:
                assert np.all(got == 0xFFFF), (label, i, "frozen tensor written")
            else:
                assert np.array_equal(got, oracle.gather_tensor(ref.op, i, params)), (label, i)
    finally:
        ref.close()
        run.close()


@pytest.mark.parametrize("name", ["tiny-world4", "odd-ds3-M3", "multi-tile-world16-M2", "tp4-world8", "world1",
                                  "world128-max", "world64-tp4-M2", "zero-size-tensors", "fp32-grads-world16"])
def test_shard_views_reproduce_the_plan_update(name):
    """check_shard_views on the named plans."""
    c = SMALL[name]
    run = Run(c)
    try:
        master0, m0, v0 = (torch.from_numpy(x).cuda() for x in run.state_host())
        run.update()
        torch.cuda.synchronize()
        check_shard_views(run, c, master0, m0, v0, name)
    finally:
        run.close()


def test_shard_view_accumulates_microbatches():
    """grs_accumulate on a shard view adds a reduced microbatch shard into
    the view's accumulator bucket by bucket, padding kept at zero."""
    g = grs()
    run = Run(SMALL["multi-tile-world16-M2"])
    try:
        view = g.grs_plan_shard_view(run.plan, 1, 1)
        try:
            vi = g.grs_plan_query(view)
            n = vi["n_state_pad"]
            gen = torch.Generator(device="cuda").manual_seed(9)
            a = torch.randn(n, generator=gen, device="cuda")
            b = torch.randn(n, generator=gen, device="cuda")
            want = a + b
            for bk in range(vi["n_buckets"]):
                d = g.grs_bucket_info(view, bk)
                lo, L, used = int(d["state_offset"]), int(d["padded"]), int(d["used"])
                want[lo + used:lo + L] = 0.0
                g.grs_accumulate(view, bk, a.data_ptr() + 4 * lo, b.data_ptr() + 4 * lo, run.stream())
            torch.cuda.synchronize()
            assert g.grs_check_device_errors(view, run.stream()) == 0
            assert torch.equal(a, want)
        finally:
            g.grs_plan_destroy(view)
    finally:
        run.close()


def test_accumulate_entry_point():
    c = SMALL["odd-ds3-M3"]
    run = Run(c)
    try:
        g = grs()
        gen = torch.Generator(device="cuda").manual_seed(3)
        run.reduce()
        torch.cuda.synchronize()
        before = run.acc.clone()
        mb = torch.randn(run.acc.numel(), generator=gen, device="cuda")
        s = run.stream()
        for b in range(run.info["n_buckets"]):
            d = g.grs_bucket_info(run.plan, b)
            g.grs_accumulate(run.plan, b, run.acc.data_ptr() + 4 * d["state_offset"],
                             mb.data_ptr() + 4 * d["state_offset"], s)
        torch.cuda.synchronize()
        pad = torch.tensor(padding_mask(run.op), device="cuda")
        want = (before[:run.nsp].double() + mb[:run.nsp].double()).float()
        want[pad] = 0
        assert torch.equal(run.acc[:run.nsp], want)
    finally:
        run.close()


def test_nonfinite_gradient_is_flagged_and_propagates():
    c = SMALL["odd-ds2"]
    run = Run(c)
    try:
        master0, m0, v0 = run.state_host()
        run.grads[0][1][3] = float("nan")  # a valid element of the RA bucket
        run.update()
        assert run.check_flags() == grs().GRS_ERR_NONFINITE
        assert run.check_flags() == 0  # flags are cleared by the check
        res = oracle_update(run, master0, m0, v0, step=1)
        assert np.isnan(res.norm_sq)
        full_check(run, res, "nan")
    finally:
        run.close()


def test_argument_errors():
    g = grs()
    c = SMALL["odd-ds2"]
    run = Run(c)
    try:
        s = run.stream()
        ptrs = run.ptrs(0)
        with pytest.raises(g.GrsError) as ei:
            g.grs_reduce_all(run.plan, [ptrs[0] + 2] + ptrs[1:], run.acc.data_ptr(), 0, 0, None, s)
        assert ei.value.status == g.GRS_ERR_ALIGNMENT
        with pytest.raises(g.GrsError) as ei:
            g.grs_reduce_all(run.plan, [None] + ptrs[1:], run.acc.data_ptr(), 0, 0, None, s)
        assert ei.value.status == g.GRS_ERR_INVALID_ARG
        with pytest.raises(g.GrsError) as ei:
            g.grs_reduce_all(run.plan, ptrs, run.acc.data_ptr() + 4, 0, 0, None, s)
        assert ei.value.status == g.GRS_ERR_ALIGNMENT
        with pytest.raises(g.GrsError) as ei:
            g.grs_reduce_all(run.plan, ptrs, run.acc.data_ptr(), 0, 1, None, s)
        assert ei.value.status == g.GRS_ERR_INVALID_ARG
        with pytest.raises(g.GrsError) as ei:
            g.grs_reduce_bucket(run.plan, 99, ptrs, run.acc.data_ptr(), 0, 0, None, s)
        assert ei.value.status == g.GRS_ERR_INVALID_ARG
        used = torch.ones(len(c.numels), dtype=torch.uint8, device="cuda")
        with pytest.raises(g.GrsError) as ei:  # norm partials need a workspace
            g.grs_reduce_all_masked(run.plan, ptrs, run.acc.data_ptr(), 0, 1, used.data_ptr(), None, s)
        assert ei.value.status == g.GRS_ERR_INVALID_ARG
        with pytest.raises(g.GrsError) as ei:
            g.grs_reduce_all_masked(run.plan, ptrs, run.acc.data_ptr(), 0, 0, None, None, s)
        assert ei.value.status == g.GRS_ERR_INVALID_ARG
        with pytest.raises(g.GrsError) as ei:
            g.grs_reduce_all_masked(run.plan, ptrs, run.acc.data_ptr(), 0, 1, used.data_ptr(),
                                    run.ws.data_ptr() + 4, s)
        assert ei.value.status == g.GRS_ERR_ALIGNMENT
        hp = g.make_adamw(1e-3, 0.9, 0.999, 1e-8, 0.0, 1.0, 0, 1)
        with pytest.raises(g.GrsError) as ei:
            g.grs_clip_adamw_step(run.plan, hp, run.norm.data_ptr(), run.acc.data_ptr(),
                                  run.master.data_ptr(), run.m.data_ptr(), run.v.data_ptr(),
                                  run.params.data_ptr(), s)
        assert ei.value.status == g.GRS_ERR_INVALID_ARG
        # ALREADY_REDUCED-only bucket needs rank 0 only
        ar = [b for b in range(run.op.n_buckets) if int(run.op.b_tag[b]) == AR][0]
        d = g.grs_bucket_info(run.plan, ar)
        g.grs_reduce_bucket(run.plan, ar, [ptrs[0] + 2 * d["rank_offset"]] + [None] * (c.world - 1),
                            run.acc.data_ptr() + 4 * d["state_offset"], 0, 0, None, s)
        assert run.check_flags() == 0
    finally:
        run.close()


@pytest.mark.parametrize("name", ["multi-tile-world16-M2", "odd-ds3-M3", "tiny-world4", "fp32-grads-world8-M3",
                                  "many-small-tensors"])
def test_step_from_host_matches_device_path(name):
    """grs_step_from_host (host gradients, pipelined copies, per-bucket
    reductions) gives the device path's results bit for bit, and reads the
    parameters and the norm back to the host; two steps in a row."""
    g = grs()
    c = SMALL[name]
    a = Run(c)
    b = Run(c)
    try:
        W, M = c.world, c.n_micro
        gdt = a.grads[0][0].dtype  # bf16, or fp32 for GRS_PLAN_FP32_GRADS plans
        host = [torch.empty(a.grads[j][k].numel(), dtype=gdt).pin_memory()
                for j in range(M) for k in range(W)]
        stage = [torch.empty(a.grads[0][0].numel(), dtype=gdt, device="cuda")
                 for _ in range(2 * W)]
        out_params = torch.empty(a.nsp, dtype=torch.int16).pin_memory()
        out_norm = torch.empty(1, dtype=torch.float64).pin_memory()
        s = b.stream()
        for step in (1, 2):
            if step == 2:
                a.fill_grads(step_seed=2)
            for j in range(M):
                for k in range(W):
                    host[j * W + k].copy_(a.grads[j][k])
            a.update()
            hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], c.max_norm, step, M)
            g.grs_step_from_host(b.plan, hp, [t.data_ptr() for t in host], [t.data_ptr() for t in stage],
                                 b.acc.data_ptr(), b.master.data_ptr(), b.m.data_ptr(), b.v.data_ptr(),
                                 b.params.data_ptr(), b.ws.data_ptr(), b.norm.data_ptr(),
                                 out_params.data_ptr(), out_norm.data_ptr(), s)
            torch.cuda.synchronize()
            assert b.check_flags() == 0
            for x, y in ((a.acc, b.acc), (a.norm, b.norm), (a.master, b.master), (a.m, b.m),
                         (a.v, b.v), (a.params, b.params)):
                assert torch.equal(x[:max(1, min(x.numel(), a.nsp))], y[:max(1, min(y.numel(), a.nsp))])
            assert torch.equal(out_params, b.params[:a.nsp].cpu())
            assert float(out_norm[0]) == float(b.norm.cpu()[0])
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("name", ["multi-tile-world16-M2", "odd-ds3-M3"])
def test_step_from_host_back_to_back(name):
    """Three grs_step_from_host calls queued without a synchronisation in
    between (each with its own host gradients and read-back buffers): the
    copies of step n+1 overlap step n's update, and every step's results
    equal the device path's bit for bit."""
    g = grs()
    c = SMALL[name]
    a = Run(c)
    b = Run(c)
    try:
        W, M = c.world, c.n_micro
        n = a.grads[0][0].numel()
        steps = 3
        host = [[torch.empty(n, dtype=torch.int16).pin_memory() for _ in range(M * W)] for _ in range(steps)]
        outp = [torch.empty(a.nsp, dtype=torch.int16).pin_memory() for _ in range(steps)]
        outn = [torch.empty(1, dtype=torch.float64).pin_memory() for _ in range(steps)]
        stage = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(2 * W)]
        want_params, want_norm = [], []
        for t in range(steps):
            if t:
                a.fill_grads(step_seed=10 + t)
            for j in range(M):
                for k in range(W):
                    host[t][j * W + k].copy_(a.grads[j][k].view(torch.int16))
            a.update()
            torch.cuda.synchronize()
            want_params.append(a.params[:a.nsp].cpu().clone())
            want_norm.append(float(a.norm.cpu()[0]))
        s = b.stream()
        for t in range(steps):
            hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], c.max_norm, t + 1, M)
            g.grs_step_from_host(b.plan, hp, [x.data_ptr() for x in host[t]], [x.data_ptr() for x in stage],
                                 b.acc.data_ptr(), b.master.data_ptr(), b.m.data_ptr(), b.v.data_ptr(),
                                 b.params.data_ptr(), b.ws.data_ptr(), b.norm.data_ptr(),
                                 outp[t].data_ptr(), outn[t].data_ptr(), s)
        torch.cuda.synchronize()
        assert b.check_flags() == 0
        for t in range(steps):
            assert torch.equal(outp[t], want_params[t]), f"step {t + 1}"
            assert float(outn[t][0]) == want_norm[t], f"step {t + 1}"
        for x, y in ((a.acc, b.acc), (a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert torch.equal(x[:a.nsp], y[:a.nsp])
    finally:
        a.close()
        b.close()


def test_frozen_tensors_excluded():
    """GRS_TENSOR_FROZEN tensors take no place in the plan: parity of the
    update on the rest, and the gather leaves their storage untouched."""
    c = Case([4096, 1000, 512 * 2, 96, 3000, 777], [RA, RA, LS, AR, PS, RA], 8, 2, 2, 2, 1 << 16, 2,
             1e-3, 41, tensor_flags=[0, 1, 0, 0, 1, 0])
    run = Run(c)
    try:
        assert grs().grs_tensor_info(run.plan, 1)["bucket"] == -1
        master0, m0, v0 = run.state_host()
        run.update()
        res = oracle_update(run, master0, m0, v0, step=1)
        full_check(run, res, "frozen")
        outs = [torch.full((n,), 7, dtype=torch.int16, device="cuda") for n in c.numels]
        grs().grs_gather_params(run.plan, run.params.data_ptr(), [t.data_ptr() for t in outs], run.stream())
        torch.cuda.synchronize()
        params = run.params[:run.nsp].cpu().numpy().view(np.uint16)
        for i, n in enumerate(c.numels):
            got = outs[i].cpu().numpy().view(np.uint16)
            if c.tensor_flags[i]:
                assert np.all(got == 7)
            else:
                assert np.array_equal(got, oracle.gather_tensor(run.op, i, params))
    finally:
        run.close()


@pytest.mark.parametrize("fp32,zeros,masked_reduce", [(False, False, False), (True, False, False),
                                                      (False, True, False), (False, False, True),
                                                      (True, True, True)])
def test_unused_tensors_masked_update(fp32, zeros, masked_reduce):
    """Three steps with per-step masks of tensors that got no gradient
    (grad None): masked norm + per-tensor-step AdamW against the oracle's
    masked update, the oracle carrying its own state and step counts.  With
    `zeros`, zero-size tensors sit between the others (empty segments the
    kernels' segment walk must step over); with `masked_reduce` the
    reduction itself skips the tiles of tensors without a gradient, whose
    accumulator is then not compared (it is unspecified)."""
    numels = [5000, 33, 4096 * 2, 17, 2048, 999, 64]
    owners = [RA, RA, LS, AR, PS, RA, LS]
    flags = [0, 0, 0, 0, 0, 1, 0]
    masks = [[1, 1, 1, 1, 1, 0, 1], [1, 0, 1, 0, 1, 0, 0], [0, 1, 1, 1, 0, 0, 1]]
    if zeros:
        # a zero-size tensor after tensors 0, 1, 2 and 4, with the owner of its neighbour
        for at in (5, 3, 2, 1):
            numels.insert(at, 0)
            owners.insert(at, owners[at - 1])
            flags.insert(at, 0)
            for mk in masks:
                mk.insert(at, at % 2)
    c = Case(numels, owners, 8, 2, 2, 2, 1 << 15, 2, 1e-3, 42, fp32_grads=fp32, tensor_flags=flags)
    run = Run(c)
    try:
        n = len(c.numels)
        steps_dev = torch.zeros(n, dtype=torch.int32, device="cuda")
        master, m, v = run.state_host()
        bits = run.params[:run.nsp].cpu().numpy().view(np.uint16).copy()
        steps = [0] * n
        for k, used in enumerate(masks):
            if k:
                run.fill_grads(step_seed=k + 1)
            used_dev = torch.tensor(used, dtype=torch.uint8, device="cuda")
            if masked_reduce:
                run.masked_reduce(used_dev)  # masked norm partials fused into the last microbatch
            else:
                run.reduce(emit=False)
            run.masked_update(used_dev, steps_dev, partials_ready=masked_reduce)
            if masked_reduce:  # the fused partials give the separate masked pass's S bit for bit
                sep = run.masked_norm_separate(used_dev)
                torch.cuda.synchronize()
                assert float(sep.cpu()[0]) == float(run.norm.cpu()[0]), (k, float(sep[0]), float(run.norm[0]))
            torch.cuda.synchronize()
            assert run.check_flags() == 0
            res, steps = oracle.full_update_masked(run.op, run.bucket_inputs, c.n_micro, c.hp, c.max_norm,
                                                   used, steps, master, m, v, bits)
            where = None
            if masked_reduce:
                where = np.ones(run.nsp, bool)
                for i in range(n):
                    if not used[i]:
                        for lo, hi in run.op.tensor_rows(i):
                            where[lo:hi] = False
            full_check(run, res, f"masked step {k + 1}", acc_where=where)
            got_steps = steps_dev.cpu().tolist()
            for i in range(n):
                if not c.tensor_flags[i]:
                    assert got_steps[i] == steps[i], (i, got_steps, steps)
            master, m, v, bits = res.master, res.m, res.v, res.params_bf16
    finally:
        run.close()


def test_masked_update_with_many_small_tensors():
    """A random half of 3000 small tensors without a gradient: nearly every
    norm and update tile spans tensors with and without one (the per-element
    segment walk, not the whole-tile shortcut)."""
    c = SMALL["many-small-tensors"]
    run = Run(c)
    try:
        n = len(c.numels)
        rng = np.random.default_rng(7)
        used = rng.integers(0, 2, n).tolist()
        steps = [0] * n
        steps_dev = torch.zeros(n, dtype=torch.int32, device="cuda")
        master, m, v = run.state_host()
        bits = run.params[:run.nsp].cpu().numpy().view(np.uint16).copy()
        run.reduce(emit=False)
        run.masked_update(torch.tensor(used, dtype=torch.uint8, device="cuda"), steps_dev)
        torch.cuda.synchronize()
        assert run.check_flags() == 0
        res, steps = oracle.full_update_masked(run.op, run.bucket_inputs, c.n_micro, c.hp, c.max_norm,
                                               used, steps, master, m, v, bits)
        full_check(run, res, "many small tensors, masked")
        assert steps_dev.cpu().tolist() == steps
    finally:
        run.close()


def random_case(rng, trial):
    """A random small plan: degrees, 1..24 tensors of all tags with 0..3000
    elements (LOCAL_SHARD a multiple of tp), bucket sizes from tiny to large,
    some tensors frozen, bf16 or fp32 gradients, 1..3 microbatches, clipping
    on or off, random AdamW hyper-parameters."""
    tp = int(rng.choice([1, 2, 3, 4]))
    dr = int(rng.choice([1, 2, 3]))
    ds = int(rng.choice([1, 2, 3, 4, 5]))
    n = int(rng.integers(1, 25))
    owners = [int(x) for x in rng.integers(0, 4, n)]
    numels = [int(rng.integers(0, 3001 // (tp if o == LS else 1))) * (tp if o == LS else 1) for o in owners]
    if sum(numels) == 0:
        numels[0] = 8 * tp
    flags = [int(x) for x in (rng.random(n) < 0.15)]
    if all(flags[i] or numels[i] == 0 for i in range(n)):
        flags = [0] * n
    bb = int(rng.choice([2, 64, 1000, 1 << 12, 1 << 20]))
    hp = (float(rng.choice([1e-3, 3e-4, 1e-2])), float(rng.choice([0.9, 0.8])), float(rng.choice([0.999, 0.95])),
          float(rng.choice([1e-8, 1e-6])), float(rng.choice([0.0, 0.01, 0.1])))
    return Case(numels, owners, tp * dr * ds, tp, dr, -1 if rng.random() < 0.2 else ds, bb,
                int(rng.integers(1, 4)), float(rng.choice([1e-3, 1e-2, 1e-1])), 500 + trial, hp=hp,
                max_norm=float(rng.choice([1.0, 0.05, 0.0])), fp32_grads=bool(rng.random() < 0.3),
                tensor_flags=flags)


@pytest.mark.parametrize("trial", range(16))
def test_random_small_plans_match_oracle(trial):
    """Random plans (random_case): one plain update against the oracle, every
    rank's shard view against it (check_shard_views) and the update writing
    per-tensor storage (check_update_to_tensors); the masked reduction, norm
    and update with a random mask against the oracle's masked update; and
    the single-launch update against the plain one, bit for bit, where its
    limits allow."""
    rng = np.random.default_rng(7000 + trial)
    c = random_case(rng, trial)
    g = grs()
    run = Run(c)
    try:
        master0, m0, v0 = run.state_host()
        bits0 = run.params[:run.nsp].cpu().numpy().view(np.uint16).copy()
        run.update()
        res = oracle_update(run, master0, m0, v0, step=1)
        full_check(run, res, f"random {trial} plain")
        check_shard_views(run, c, *(torch.from_numpy(x).cuda() for x in (master0, m0, v0)), f"random {trial}")
    finally:
        run.close()
    check_update_to_tensors(c, f"random {trial}")
    n = len(c.numels)
    used = [int(x) for x in (rng.random(n) < 0.7)]
    mrun = Run(c)
    try:
        used_dev = torch.tensor(used, dtype=torch.uint8, device="cuda")
        mrun.masked_reduce(used_dev)
        mrun.masked_update(used_dev, torch.zeros(n, dtype=torch.int32, device="cuda"), partials_ready=True)
        sep = mrun.masked_norm_separate(used_dev)
        torch.cuda.synchronize()
        assert mrun.check_flags() == 0
        assert float(sep.cpu()[0]) == float(mrun.norm.cpu()[0]), (trial, float(sep[0]), float(mrun.norm[0]))
        res, _ = oracle.full_update_masked(mrun.op, mrun.bucket_inputs, c.n_micro, c.hp, c.max_norm, used, [0] * n,
                                           master0, m0, v0, bits0)
        where = np.ones(mrun.nsp, bool)
        for i in range(n):
            if not used[i]:
                for lo, hi in mrun.op.tensor_rows(i):
                    where[lo:hi] = False
        full_check(mrun, res, f"random {trial} masked", acc_where=where)
    finally:
        mrun.close()
    a, b = Run(c), Run(c)
    try:
        rows = sum(a.op.copies(bk) for bk in range(a.op.n_buckets))
        if (a.info["n_reduce_tiles"] > g.GRS_SMALL_MAX_TILES or rows > g.GRS_SMALL_MAX_TILES or
                c.n_micro * c.world > g.GRS_SMALL_MAX_BUFFERS):
            return
        a.update()
        hp = g.make_adamw(*c.hp, c.max_norm, 1, c.n_micro)
        norm = torch.zeros(1, dtype=torch.float64, device="cuda")
        g.grs_update_small(b.plan, hp, [p for j in range(c.n_micro) for p in b.ptrs(j)], b.acc.data_ptr(),
                           b.master.data_ptr(), b.m.data_ptr(), b.v.data_ptr(), b.params.data_ptr(),
                           norm.data_ptr(), b.stream())
        torch.cuda.synchronize()
        assert a.check_flags() == 0 and b.check_flags() == 0
        assert torch.equal(a.norm, norm)
        for nm in ("acc", "master", "m", "v", "params"):
            assert torch.equal(getattr(a, nm)[:a.nsp], getattr(b, nm)[:b.nsp]), nm
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("trial", [3, 10, 17, 26, 33, 39])
def test_random_medium_plans_match_oracle(trial):
    """Random plans of up to 300k-element tensors (many tiles per bucket
    row, every tag, bf16 or fp32 gradients, 1..3 microbatches, degrees up to
    tp 4 x dp_replicate 2 x dp_shard 8): one update against the oracle, with
    the shard views and the per-tensor write checked as on the small plans.
    Seed 10 meets an ill-conditioned AdamW point (fp32 gradients cancelling
    across microbatches to 1.7e-9), where the check follows the bracket."""
    rng = np.random.default_rng(90000 + trial)
    tp = int(rng.choice([1, 2, 4]))
    dr = int(rng.choice([1, 2]))
    ds = int(rng.choice([1, 2, 4, 8]))
    n = int(rng.integers(1, 12))
    owners = [int(x) for x in rng.integers(0, 4, n)]
    numels = [int(rng.integers(0, 300000 // (tp if o == LS else 1))) * (tp if o == LS else 1) for o in owners]
    if sum(numels) == 0:
        numels[0] = 8 * tp
    c = Case(numels, owners, tp * dr * ds, tp, dr, ds, int(rng.choice([1 << 14, 1 << 18, 1 << 22])),
             int(rng.integers(1, 4)), 1e-3, 800 + trial, fp32_grads=bool(rng.random() < 0.3))
    run = Run(c)
    try:
        master0, m0, v0 = run.state_host()
        run.update()
        res = oracle_update(run, master0, m0, v0, step=1)
        full_check(run, res, f"medium {trial}")
        check_shard_views(run, c, *(torch.from_numpy(x).cuda() for x in (master0, m0, v0)), f"medium {trial}")
    finally:
        run.close()
    check_update_to_tensors(c, f"medium {trial}")


def test_masked_reduction_skips_tiles_of_unused_tensors():
    """The masked reduction neither reads nor writes the tiles that lie wholly
    in tensors without a gradient: with those tensors' gradients poisoned
    (NaN in every rank buffer) and the accumulator pre-filled, their whole
    tiles keep the fill, every used tensor's accumulator equals the plain
    reduction of clean inputs bit for bit, and the masked norm stays finite."""
    c = Case([300000, 1024, 65536 * 4, 4099, 200000, 70002], [RA, PS, LS, AR, RA, LS], 8, 2, 2, 2, 1 << 18, 1,
             1e-3, 61)
    a, b = Run(c), Run(c)
    try:
        g = grs()
        n = len(c.numels)
        used = [1, 1, 0, 1, 0, 1]
        used_dev = torch.tensor(used, dtype=torch.uint8, device="cuda")
        a.reduce(emit=False)
        op = b.op
        for i in range(n):  # poison the unused tensors' gradients on every rank
            if used[i]:
                continue
            bk = int(op.t_bucket[i])
            lo = int(op.b_rank_off[bk]) + int(op.t_offset[i])
            for k in range(c.world):
                b.grads[0][k].view(torch.int16)[lo:lo + op.per_rank(i)] = 0x7FC0
        b.acc.fill_(123.0)
        b.masked_reduce(used_dev, emit=False)
        torch.cuda.synchronize()
        assert b.check_flags() == 0
        got, want = b.acc[:b.nsp].cpu().numpy(), a.acc[:a.nsp].cpu().numpy()
        untouched = 0
        for i in range(n):
            for lo, hi in op.tensor_rows(i):
                if used[i]:
                    assert np.array_equal(got[lo:hi], want[lo:hi]), i
                else:
                    untouched += int((got[lo:hi] == 123.0).sum())
        assert untouched > 0.9 * sum(c.numels[i] for i in range(n) if not used[i])
        b.masked_update(used_dev, torch.zeros(n, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        assert b.check_flags() == 0
        assert np.isfinite(float(b.norm.cpu()[0]))
        # The same reduction with the norm partials fused: the poisoned
        # elements of tiles shared with used tensors count as zero there too.
        b.acc.fill_(123.0)
        b.masked_reduce(used_dev)
        b.norm_sq(partials_ready=True)
        fused = b.norm.clone()
        sep = b.masked_norm_separate(used_dev)
        torch.cuda.synchronize()
        assert b.check_flags() == 0
        assert np.isfinite(float(fused.cpu()[0])) and float(fused.cpu()[0]) == float(sep.cpu()[0])
    finally:
        a.close()
        b.close()


def test_masked_reduction_with_every_tensor_used_equals_plain():
    """grs_reduce_all_masked with every tensor marked used reduces every tile:
    the accumulator and the fused norm partials (hence S) equal
    grs_reduce_all's bit for bit (two microbatches)."""
    c = SMALL["multi-tile-world16-M2"]
    a, b = Run(c), Run(c)
    try:
        g = grs()
        ones = torch.ones(len(c.numels), dtype=torch.uint8, device="cuda")
        a.reduce(emit=True)
        a.norm_sq(partials_ready=True)
        b.masked_reduce(ones)
        b.norm_sq(partials_ready=True)
        torch.cuda.synchronize()
        assert a.check_flags() == 0 and b.check_flags() == 0
        assert torch.equal(a.acc[:a.nsp], b.acc[:b.nsp])
        assert float(a.norm.cpu()[0]) == float(b.norm.cpu()[0])
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("hint", ["matching", "none"])
def test_masked_path_with_every_tensor_used_equals_plain_path(hint):
    """With every tensor marked as having a gradient, the masked norm and the
    per-tensor-step AdamW produce the plain path's norm, master, moments and
    bf16 parameters bit for bit, over three steps (the masked norm replays
    the same per-tile order; the per-tensor factors equal the plan-wide
    ones), whether the factors come from the host (the caller's step equals
    every tensor's) or are computed on the device (no step given)."""
    c = SMALL["multi-tile-world16-M2"]
    a, b = Run(c), Run(c)
    try:
        n = len(c.numels)
        ones = torch.ones(n, dtype=torch.uint8, device="cuda")
        steps = torch.zeros(n, dtype=torch.int32, device="cuda")
        for k in range(3):
            if k:
                a.fill_grads(step_seed=k + 1)
                b.fill_grads(step_seed=k + 1)
            a.update()
            b.reduce(emit=False)
            b.masked_update(ones, steps, step_hint=k + 1 if hint == "matching" else 0)
            torch.cuda.synchronize()
            assert a.check_flags() == 0 and b.check_flags() == 0
            for name in ("acc", "norm", "master", "m", "v", "params"):
                assert torch.equal(getattr(a, name), getattr(b, name)), (k + 1, name)
        assert steps.cpu().tolist() == [3] * n
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("name", ["tiny-world4", "odd-ds2", "odd-ds3-M3", "world1", "world3-non-pow2",
                                  "world6-auto-shard", "zero-size-tensors", "fp32-grads-world8-M3", "tp4-world8",
                                  "world64-tp4-M2", "multi-tile-world16-M2"])
def test_single_launch_update_equals_three_calls(name):
    """grs_update_small (one cluster launch: reductions of every microbatch,
    norm, clip + AdamW) gives the accumulator, norm, master, moments and bf16
    parameters of grs_reduce_all + grs_grad_norm_sq + grs_clip_adamw_step
    bit for bit, over three steps; plans beyond its limits are refused."""
    g = grs()
    c = SMALL[name]
    a, b = Run(c), Run(c)
    try:
        bufs = lambda r: [p for j in range(c.n_micro) for p in r.ptrs(j)]
        norm = torch.zeros(1, dtype=torch.float64, device="cuda")
        if a.info["n_reduce_tiles"] > g.GRS_SMALL_MAX_TILES or c.n_micro * c.world > g.GRS_SMALL_MAX_BUFFERS:
            hp = g.make_adamw(*c.hp, c.max_norm, 1, c.n_micro)
            with pytest.raises(g.GrsError) as ei:
                g.grs_update_small(b.plan, hp, bufs(b), b.acc.data_ptr(), b.master.data_ptr(), b.m.data_ptr(),
                                   b.v.data_ptr(), b.params.data_ptr(), norm.data_ptr(), b.stream())
            assert ei.value.status == g.GRS_ERR_SHAPE
            return
        for step in range(1, 4):
            if step > 1:
                a.fill_grads(step_seed=step)
                b.fill_grads(step_seed=step)
            a.update()
            hp = g.make_adamw(*c.hp, c.max_norm, step, c.n_micro)
            g.grs_update_small(b.plan, hp, bufs(b), b.acc.data_ptr(), b.master.data_ptr(), b.m.data_ptr(),
                               b.v.data_ptr(), b.params.data_ptr(), norm.data_ptr(), b.stream())
            torch.cuda.synchronize()
            assert a.check_flags() == 0 and b.check_flags() == 0
            assert torch.equal(a.norm, norm), (step, float(a.norm[0]), float(norm[0]))
            for nm in ("acc", "master", "m", "v", "params"):
                assert torch.equal(getattr(a, nm)[:a.nsp], getattr(b, nm)[:b.nsp]), (step, nm)
    finally:
        a.close()
        b.close()


def test_trailing_accumulation_window():
    """A window that ends after 3 of 4 microbatches: the update averages the
    3 accumulated microbatches (G = acc / 3)."""
    c = SMALL["multi-tile-world16-M2"]
    c = Case(c.numels, c.owners, c.world, c.tp, c.dp_replicate, c.dp_shard, c.bucket_bytes, 4,
             c.grad_std, 43)
    run = Run(c)
    try:
        master0, m0, v0 = run.state_host()
        g = grs()
        run.reduce(n_micro=3)
        g.grs_grad_norm_sq(run.plan, run.acc.data_ptr(), 3, run.ws.data_ptr(), 1, run.norm.data_ptr(),
                           run.stream())
        hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], c.max_norm, 1, 3)
        g.grs_clip_adamw_step(run.plan, hp, run.norm.data_ptr(), run.acc.data_ptr(), run.master.data_ptr(),
                              run.m.data_ptr(), run.v.data_ptr(), run.params.data_ptr(), run.stream())
        res = oracle.full_update(run.op, lambda b: run.bucket_inputs(b)[:3], 3, c.hp, c.max_norm, 1,
                                 master0, m0, v0, bounds=True)
        full_check(run, res, "trailing window")
    finally:
        run.close()


def test_bounded_wait_times_out_and_context_survives():
    """A device wait that nothing completes gives up after its limit, the
    plan reports GRS_ERR_TIMEOUT, and the next update still runs correctly."""
    g = grs()
    c = SMALL["odd-ds2"]
    run = Run(c)
    try:
        import time
        t0 = time.time()
        g.grs_selftest_bounded_wait(run.plan, 20_000_000, run.stream())  # 20 ms
        assert run.check_flags() == g.GRS_ERR_TIMEOUT
        assert time.time() - t0 < 5.0
        assert run.check_flags() == 0
        with pytest.raises(g.GrsError):
            g.grs_selftest_bounded_wait(run.plan, 10, run.stream())
        master0, m0, v0 = run.state_host()
        run.update()
        assert run.check_flags() == 0
        full_check(run, oracle_update(run, master0, m0, v0, step=1), "after timeout")
    finally:
        run.close()


def test_overlapped_reverse_order_reduction_matches_grouped():
    """Buckets produced in reverse order on a 'backward' stream, each reduced
    on a side stream as soon as its event fires, with a capped grid: the
    accumulator and the norm equal the grouped launch's bit for bit, and the
    whole update matches the oracle ("refactor(distributed): establish
    shared native TP replica ownership", "Preserved prototype and evidence":
    the asynchronous FP32 reduction hook; "Proposed scope": overlap during
    backward)."""
    g = grs()
    c = SMALL["multi-tile-world16-M2"]
    ref = Run(c)
    run = Run(c)
    try:
        master0, m0, v0 = run.state_host()
        ref.update()
        torch.cuda.synchronize()
        src = [[t.clone() for t in mb] for mb in run.grads]
        for mb in run.grads:
            for t in mb:
                t.fill_(float("nan"))  # gradients do not exist yet
        torch.cuda.synchronize()
        producer = torch.cuda.Stream()
        side = torch.cuda.Stream()
        nb = run.info["n_buckets"]
        for j in range(c.n_micro):
            for b in reversed(range(nb)):
                d = g.grs_bucket_info(run.plan, b)
                lo, hi = d["rank_offset"], d["rank_offset"] + d["padded"]
                ev = torch.cuda.Event()
                with torch.cuda.stream(producer):
                    for k in range(c.world):
                        run.grads[j][k][lo:hi].copy_(src[j][k][lo:hi])
                    ev.record(producer)
                rp = [t.data_ptr() + 2 * d["rank_offset"] for t in run.grads[j]]
                g.grs_reduce_bucket_ex(run.plan, b, rp, run.acc.data_ptr() + 4 * d["state_offset"], int(j > 0),
                                       int(j == c.n_micro - 1), run.ws.data_ptr(), 16, ev.cuda_event,
                                       side.cuda_stream)
        with torch.cuda.stream(side):
            g.grs_grad_norm_sq(run.plan, run.acc.data_ptr(), c.n_micro, run.ws.data_ptr(), 1,
                               run.norm.data_ptr(), side.cuda_stream)
            hp = g.make_adamw(c.hp[0], c.hp[1], c.hp[2], c.hp[3], c.hp[4], c.max_norm, 1, c.n_micro)
            g.grs_clip_adamw_step(run.plan, hp, run.norm.data_ptr(), run.acc.data_ptr(), run.master.data_ptr(),
                                  run.m.data_ptr(), run.v.data_ptr(), run.params.data_ptr(), side.cuda_stream)
        torch.cuda.synchronize()
        for x, y in ((ref.acc, run.acc), (ref.norm, run.norm), (ref.master, run.master), (ref.params, run.params)):
            assert torch.equal(x, y)
        assert run.check_flags() == 0
        full_check(run, oracle_update(run, master0, m0, v0, step=1), "overlapped reverse order")
    finally:
        ref.close()
        run.close()


def test_check_already_reduced_flags_disagreeing_copies():
    g = grs()
    c = Case([4096, 999, 777, 64 * 2], [RA, AR, AR, LS], 4, 2, 1, 2, 1 << 20, 1, 1e-2, 61)
    run = Run(c)
    try:
        s = run.stream()
        for b in range(run.op.n_buckets):  # make every AR copy equal rank 0's
            if int(run.op.b_tag[b]) == AR:
                ro, used = int(run.op.b_rank_off[b]), int(run.op.b_used[b])
                for k in range(1, c.world):
                    run.grads[0][k][ro:ro + used] = run.grads[0][0][ro:ro + used]
        g.grs_check_already_reduced(run.plan, run.ptrs(0), s)
        assert run.check_flags() == 0
        ar = [b for b in range(run.op.n_buckets) if int(run.op.b_tag[b]) == AR][0]
        e = int(run.op.b_rank_off[ar]) + int(run.op.b_used[ar]) - 1  # last valid element
        run.grads[0][3][e] = run.grads[0][3][e] + 1.0
        g.grs_check_already_reduced(run.plan, run.ptrs(0), s)
        assert run.check_flags() == g.GRS_ERR_INVALID_ARG
        assert "ALREADY_REDUCED" in g.grs_last_error()
        assert run.check_flags() == 0
    finally:
        run.close()


@pytest.mark.parametrize("kind", ["every-tensor-frozen", "every-tensor-empty"])
def test_plans_without_state(kind):
    """Degenerate plans with no state element: every tensor frozen (no
    bucket at all) or every tensor of size zero (buckets without tiles).
    Every entry point of the path runs and does nothing: S = 0 as the
    oracle's, no device flag, and the caller's buffers untouched."""
    g = grs()
    numels = [100, 200, 64] if kind == "every-tensor-frozen" else [0, 0, 0]
    flags = [1, 1, 1] if kind == "every-tensor-frozen" else [0, 0, 0]
    c = Case(numels, [RA, PS, AR], 4, 1, 2, 2, 1 << 20, 2, 1e-3, 31, tensor_flags=flags)
    run = Run(c)
    try:
        assert run.nsp == 0 and run.info["n_reduce_tiles"] == 0
        s = run.stream()
        run.master.fill_(0.5)
        run.norm.fill_(7.0)
        run.update()
        torch.cuda.synchronize()
        assert run.check_flags() == 0
        res = oracle_update(run, np.zeros(0, np.float32), np.zeros(0, np.float32), np.zeros(0, np.float32), step=1)
        assert float(run.norm.cpu()[0]) == 0.0 == float(res.norm_sq)
        used = torch.ones(len(numels), dtype=torch.uint8, device="cuda")
        steps = torch.zeros(len(numels), dtype=torch.int32, device="cuda")
        run.norm.fill_(7.0)
        run.masked_reduce(used)
        run.masked_update(used, steps, partials_ready=True)
        torch.cuda.synchronize()
        assert run.check_flags() == 0 and float(run.norm.cpu()[0]) == 0.0
        # tensors without state keep their step counts (frozen ones are ignored)
        assert steps.cpu().tolist() == ([0, 0, 0] if kind == "every-tensor-frozen" else [1, 1, 1])
        dst = [torch.full((max(n, 1),), -3, dtype=torch.int16, device="cuda") for n in numels]
        g.grs_gather_params(run.plan, run.params.data_ptr(), [t.data_ptr() for t in dst], s)
        logical = torch.full((8,), -1.0, dtype=torch.float32, device="cuda")
        g.grs_state_to_logical(run.plan, run.master.data_ptr(), logical.data_ptr(), s)
        g.grs_state_from_logical(run.plan, logical.data_ptr(), run.m.data_ptr(), s)
        hp = g.make_adamw(*c.hp, c.max_norm, 1, c.n_micro)
        run.norm.fill_(7.0)
        g.grs_update_small(run.plan, hp, [p for j in range(c.n_micro) for p in run.ptrs(j)], run.acc.data_ptr(),
                           run.master.data_ptr(), run.m.data_ptr(), run.v.data_ptr(), run.params.data_ptr(),
                           run.norm.data_ptr(), s)
        torch.cuda.synchronize()
        assert run.check_flags() == 0 and float(run.norm.cpu()[0]) == 0.0
        assert all(bool((t == -3).all()) for t in dst)
        assert bool((logical == -1.0).all()) and bool((run.master == 0.5).all())
    finally:
        run.close()
