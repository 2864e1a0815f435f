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
from gpu_support import (Case, Run, assert_bf16_cast, assert_close, case_from_workload, grs,
                         oracle_update, padding_mask)

pytestmark = pytest.mark.gpu

RA, PS, LS, AR = 0, 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.init()


def full_check(run: Run, res, what=""):
    torch.cuda.synchronize()
    n = run.nsp
    pad = padding_mask(run.op)
    acc = run.acc[:n].cpu().numpy()
    assert_close(acc, res.acc, f"{what} acc")
    assert np.all(acc[pad] == 0), f"{what} acc padding not zero"
    norm = float(run.norm.cpu()[0])
    assert_close([norm], [res.norm_sq], f"{what} norm_sq")
    master, m, v = run.state_host()
    assert_close(master, res.master, f"{what} master")
    assert_close(m, res.m, f"{what} m")
    assert_close(v, res.v, f"{what} v")
    for name, arr in (("master", master), ("m", m), ("v", v)):
        assert np.all(arr[pad] == 0), f"{what} {name} padding not zero"
    bits = run.params[:n].cpu().numpy().view(np.uint16)
    assert_bf16_cast(bits, master, res.params_bf16, res.master, f"{what} params")
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
    for name in ("tiny-world4", "odd-ds3-M3", "multi-tile-world16-M2"):
        c = SMALL[name]
        run = Run(c)
        try:
            run.update()
            torch.cuda.synchronize()
            outs = [torch.full((max(n, 1),), -1, dtype=torch.int16, device="cuda") for n in c.numels]
            # odd offsets inside a larger buffer exercise the unaligned paths
            big = torch.full((sum(c.numels) + 64,), -1, dtype=torch.int16, device="cuda")
            ptrs, views, off = [], [], 3
            for n in c.numels:
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


@pytest.mark.parametrize("name", ["multi-tile-world16-M2", "odd-ds3-M3", "tiny-world4"])
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
        host = [torch.empty(a.grads[j][k].numel(), dtype=torch.int16).pin_memory()
                for j in range(M) for k in range(W)]
        stage = [torch.empty(a.grads[0][0].numel(), dtype=torch.bfloat16, device="cuda")
                 for _ in range(2 * W)]
        out_params = torch.empty(a.nsp, dtype=torch.int16).pin_memory()
        out_norm = torch.empty(1, dtype=torch.float64).pin_memory()
        s = b.stream()
        for step in (1, 2):
            if step == 2:
                a.fill_grads(step_seed=2)
            for j in range(M):
                for k in range(W):
                    host[j * W + k].copy_(a.grads[j][k].view(torch.int16))
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
